// la_api.cu -- the extern "C" entry points of the seg_la library (declared in include/la.h):
// host-side argument checks, the per-device error word, and kernel dispatch.  No entry point
// allocates device memory or synchronises, except la_poll_error, which synchronises by design.
#include <math.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "la.h"
#include "la_extend_bal.h"
#include "la_internal.h"

namespace {

// The extend kernel runs one CTA per (request, head, segment) (la_extend_w.cu).
constexpr int kExtendCtasPerHead = 1;

// Per-device error word: kernels OR bits into it when they find a fault the host cannot see
// (out-of-range slot, inconsistent cu_seqlens, a bounded wait that ran out).  Module-scope
// device variable; its address is looked up once per device and passed to kernels.
__device__ unsigned int g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned int *g_err_ptr[kMaxDevices] = {nullptr};
std::atomic<unsigned long long> g_wait_limit{0};
std::atomic<int> g_column_split{1};
std::atomic<int> g_persistent{1};
std::atomic<int> g_balanced{1};

// Default bound on a device wait: far above any legitimate wait inside one CTA (microseconds),
// short enough that a lost arrival ends the kernel in about two seconds instead of hanging.
constexpr unsigned long long kDefaultWaitLimitUs = 2000000ull;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// int32, fp32 and uint8 arrays are read element by element: 4-byte alignment (1 for uint8)
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

la_status error_word_ptr(unsigned int **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return LA_ERR_CUDA;
        g_err_ptr[dev] = static_cast<unsigned int *>(p);
    }
    *out = g_err_ptr[dev];
    return LA_OK;
}

la_status launch_status(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

int g_num_sms[kMaxDevices] = {0};

la_status num_sms(int *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return LA_ERR_CUDA;
        g_num_sms[dev] = n;
    }
    *out = g_num_sms[dev];
    return LA_OK;
}

}  // namespace

extern "C" {

const char *la_status_string(la_status status) {
    switch (status) {
        case LA_OK: return "LA_OK";
        case LA_ERR_INVALID: return "LA_ERR_INVALID: invalid argument";
        case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED: unsupported configuration";
        case LA_ERR_CUDA: return "LA_ERR_CUDA: CUDA runtime or launch error";
        case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a bounded device wait ran out";
        case LA_ERR_DEVICE_INPUT:
            return "LA_ERR_DEVICE_INPUT: a device-side index (slot, cu_seqlens, parent, accept "
                   "or track entry) was out of range";
    }
    return "LA_ERR_UNKNOWN";
}

la_status la_slopes(int H, int layer_id, int L, float *host_out) {
    if (H < 1 || L < 1 || layer_id < 0 || layer_id >= L || host_out == nullptr)
        return LA_ERR_INVALID;
    // Per-layer factor from the page's slope rule; ALiBi geometric base 2^(-8 (i+1) / H).
    const double factor =
        (L == 1) ? (1.0 + 1e-5) : (1.0 - (double)layer_id / (double)(L - 1) + 1e-5);
    for (int i = 0; i < H; ++i)
        host_out[i] = (float)(exp2(-8.0 * (double)(i + 1) / (double)H) * factor);
    return LA_OK;
}

void la_set_wait_limit(uint64_t microseconds) { g_wait_limit.store(microseconds); }

void la_set_column_split(int enable) { g_column_split.store(enable ? 1 : 0); }

void la_set_persistent(int enable) { g_persistent.store(enable ? 1 : 0); }

void la_set_balanced(int enable) { g_balanced.store(enable ? 1 : 0); }

la_status la_poll_error(la_stream stream) {
    // The error word is per device, so every kernel that may write it -- on any stream of the
    // device -- has to be finished before it is read: synchronise the stream given (which may
    // belong to another context's default) and then the whole device.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return LA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return LA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    unsigned int *err = nullptr;
    la_status st = error_word_ptr(&err);
    if (st != LA_OK) return st;
    unsigned int word = 0;
    if (cudaMemcpy(&word, err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LA_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return LA_ERR_CUDA;
    }
    if (word & la::ERR_BIT_TIMEOUT) return LA_ERR_TIMEOUT;
    if (word & (la::ERR_BIT_SLOT_RANGE | la::ERR_BIT_SEQLENS | la::ERR_BIT_PARENTS |
                la::ERR_BIT_ACCEPT | la::ERR_BIT_TRACK))
        return LA_ERR_DEVICE_INPUT;
    return LA_OK;
}

la_status la_decode(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                    float *state_pool, int num_slots, const int32_t *state_idx, la_bf16 *out,
                    int B, int H, int D, la_stream stream) {
    if (B < 0 || H < 1 || D < 1 || num_slots < 1) return LA_ERR_INVALID;
    if (D != la::kHeadDim) return LA_ERR_UNSUPPORTED;
    if (B == 0) return LA_OK;
    if (!q || !k || !v || !slopes || !state_pool || !state_idx || !out) return LA_ERR_INVALID;
    // the kernel moves q, k, v, the states and out with 16-byte vector accesses
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state_pool) ||
        !aligned16(out) || !aligned4(slopes) || !aligned4(state_idx))
        return LA_ERR_INVALID;
    la::RecurParams p{};
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    p.k = reinterpret_cast<const __nv_bfloat16 *>(k);
    p.v = reinterpret_cast<const __nv_bfloat16 *>(v);
    p.slopes = slopes;
    p.pool = state_pool;
    p.state_idx = state_idx;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.B = B;
    p.H = H;
    p.N = 1;
    p.num_slots = num_slots;
    la_status st = error_word_ptr(&p.err);
    if (st != LA_OK) return st;
    return launch_status(la::launch_recurrent(la::RECUR_DECODE, p, static_cast<cudaStream_t>(stream)));
}

la_status la_verify_chain(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v,
                          const float *slopes, const float *state_pool, int num_slots,
                          const int32_t *state_idx, float *inter_states, la_bf16 *out, int B,
                          int N, int H, int D, la_stream stream) {
    if (B < 0 || N < 1 || H < 1 || D < 1 || num_slots < 1) return LA_ERR_INVALID;
    if (D != la::kHeadDim) return LA_ERR_UNSUPPORTED;
    if ((long long)B * N > 0x7fffffffLL) return LA_ERR_INVALID;
    if (B == 0) return LA_OK;
    if (!q || !k || !v || !slopes || !state_pool || !state_idx || !inter_states || !out)
        return LA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state_pool) ||
        !aligned16(inter_states) || !aligned16(out) || !aligned4(slopes) || !aligned4(state_idx))
        return LA_ERR_INVALID;
    la::RecurParams p{};
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    p.k = reinterpret_cast<const __nv_bfloat16 *>(k);
    p.v = reinterpret_cast<const __nv_bfloat16 *>(v);
    p.slopes = slopes;
    p.pool = const_cast<float *>(state_pool);  // read only in verify mode
    p.state_idx = state_idx;
    p.inter = inter_states;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.B = B;
    p.H = H;
    p.N = N;
    p.num_slots = num_slots;
    la_status st = error_word_ptr(&p.err);
    if (st != LA_OK) return st;
    return launch_status(la::launch_recurrent(la::RECUR_VERIFY, p, static_cast<cudaStream_t>(stream)));
}

la_status la_verify_tree(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v,
                         const float *slopes, const float *state_pool, int num_slots,
                         const int32_t *state_idx, const int32_t *parents, float *inter_states,
                         la_bf16 *out, int B, int N, int H, int D, la_stream stream) {
    if (B < 0 || N < 1 || H < 1 || D < 1 || num_slots < 1) return LA_ERR_INVALID;
    if (D != la::kHeadDim) return LA_ERR_UNSUPPORTED;
    if ((long long)B * N > 0x7fffffffLL) return LA_ERR_INVALID;
    if (B == 0) return LA_OK;
    if (!q || !k || !v || !slopes || !state_pool || !state_idx || !parents || !inter_states || !out)
        return LA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state_pool) ||
        !aligned16(inter_states) || !aligned16(out) || !aligned4(slopes) || !aligned4(state_idx) ||
        !aligned4(parents))
        return LA_ERR_INVALID;
    la::RecurParams p{};
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    p.k = reinterpret_cast<const __nv_bfloat16 *>(k);
    p.v = reinterpret_cast<const __nv_bfloat16 *>(v);
    p.slopes = slopes;
    p.pool = const_cast<float *>(state_pool);  // read only in tree mode
    p.state_idx = state_idx;
    p.parents = parents;
    p.inter = inter_states;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.B = B;
    p.H = H;
    p.N = N;
    p.num_slots = num_slots;
    la_status st = error_word_ptr(&p.err);
    if (st != LA_OK) return st;
    return launch_status(la::launch_recurrent(la::RECUR_TREE, p, static_cast<cudaStream_t>(stream)));
}

la_status la_commit_accepted(const float *inter_states, const int32_t *accept_idx,
                             float *state_pool, int num_slots, const int32_t *state_idx, int B,
                             int N, int H, int D, la_stream stream) {
    if (B < 0 || N < 1 || H < 1 || D < 1 || num_slots < 1) return LA_ERR_INVALID;
    if (D != la::kHeadDim) return LA_ERR_UNSUPPORTED;
    if (B == 0) return LA_OK;
    if (!inter_states || !accept_idx || !state_pool || !state_idx) return LA_ERR_INVALID;
    if (!aligned16(inter_states) || !aligned16(state_pool) || !aligned4(accept_idx) ||
        !aligned4(state_idx))
        return LA_ERR_INVALID;
    la::CommitParams p{};
    p.inter = inter_states;
    p.accept_idx = accept_idx;
    p.pool = state_pool;
    p.state_idx = state_idx;
    p.B = B;
    p.N = N;
    p.H = H;
    p.num_slots = num_slots;
    la_status st = error_word_ptr(&p.err);
    if (st != LA_OK) return st;
    return launch_status(la::launch_commit(p, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Scratch of an extend call: the split plan's block states and initial-state copies, and for a
// grouped call (Hkv < H) at least the initial-state copies.
struct ExtendScratch {
    la::SplitPlan plan;        // seg_len == 0: no sequence split
    unsigned long long full;   // bytes with the split, before the order array
    unsigned long long copies; // bytes of the initial-state copies alone (grouped calls)
    unsigned long long order;  // bytes of the longest-first order array (large batches), after
                               // `full`
    unsigned long long recs;   // bytes of the persistent extend's request records (batches of
                               // more than one wave), after the order array
    unsigned long long bal;    // bytes of the balanced extend's plan (one-wave batches without a
                               // sequence split), after the records
};

// A one-wave batch runs balanced when its longest request (max_seqlen) is at least this many times
// the mean length T / B.  Balancing reads the keys and values before each cut a second time and
// keeps every SM streaming, which slows each chunk (3.4-3.6 us against 3.05 us); on batches of
// lengths within a factor of about two of each other the column split does as well or better.
constexpr long long kBalancedSkew = 2;

// Up to this many requests every extend CTA ranks the batch itself; above it, a pre-pass ranks
// it once into the workspace.
constexpr int kInCtaRankedRequests = 256;

la_status extend_scratch(int B, int T, int H, int Hkv, int max_seqlen, ExtendScratch *out) {
    *out = ExtendScratch{la::SplitPlan{0, 0, 1, 0, 0ull}, 0ull, 0ull, 0ull, 0ull, 0ull};
    const unsigned long long mat = (unsigned long long)la::kHeadDim * la::kHeadDim * sizeof(float);
    if (Hkv < H) out->copies = (unsigned long long)B * Hkv * mat;
    out->full = out->copies;
    if (B == 0 || T == 0) return LA_OK;
    if (B > kInCtaRankedRequests && B <= la::kMaxRankedRequests)
        out->order = ((unsigned long long)B * sizeof(int32_t) + 15ull) & ~15ull;
    int sms = 0;
    la_status st = num_sms(&sms);
    if (st != LA_OK) return st;
    if (Hkv == H && (long long)B * H > sms && B <= la::kMaxRankedRequests)
        out->recs = (unsigned long long)B * sizeof(la::ItemRec);
    const la::SplitPlan pl = la::plan_split(B, H, max_seqlen, sms, kExtendCtasPerHead);
    if (pl.seg_len > 0) {
        out->plan = pl;
        out->full = (unsigned long long)B * Hkv * (unsigned long long)(1 + pl.nblk) * mat;
    } else if (Hkv == H && B >= 2 && B <= la::kMaxBalRequests && (long long)B * H <= sms &&
               (long long)max_seqlen * B >= kBalancedSkew * (long long)T) {
        out->bal = la::bal_scratch_bytes(B, H);
    }
    return LA_OK;
}

la_status extend_impl(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                      float *state_pool, int num_slots, const int32_t *state_idx,
                      const int32_t *cu_seqlens, const uint8_t *prefix_mask,
                      const int32_t *track_lens, const int32_t *track_state_idx, la_bf16 *out,
                      long long out_rs, long long out_hs, int B, int T, int H, int Hkv, int D,
                      int max_seqlen, void *workspace, size_t workspace_bytes, la_stream stream) {
    if (B < 0 || T < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || D < 1 || num_slots < 1 ||
        max_seqlen < 0)
        return LA_ERR_INVALID;
    if (D != la::kHeadDim) return LA_ERR_UNSUPPORTED;
    // output layout: 16-byte aligned rows and heads that do not overlap (rows of heads, or heads
    // of rows), all inside the 2^40-element range the kernels index
    if (out_rs == 0) out_rs = (long long)H * D;
    if (out_hs == 0) out_hs = D;
    if (out_rs < 0 || out_hs < 0 || out_rs % 8 != 0 || out_hs % 8 != 0) return LA_ERR_INVALID;
    if (out_rs < (long long)(H - 1) * out_hs + D && out_hs < (long long)(T > 0 ? T - 1 : 0) * out_rs + D)
        return LA_ERR_INVALID;
    if (out_rs >= (1ll << 40) || out_hs >= (1ll << 40) ||
        (long long)(T > 0 ? T - 1 : 0) * out_rs + (long long)(H - 1) * out_hs + D >= (1ll << 40))
        return LA_ERR_UNSUPPORTED;
    if (B == 0) return LA_OK;
    if (!slopes || !state_pool || !state_idx || !cu_seqlens || !prefix_mask) return LA_ERR_INVALID;
    if (T > 0 && (!q || !k || !v || !out)) return LA_ERR_INVALID;
    if ((long long)T * H * D >= (1ll << 40)) return LA_ERR_UNSUPPORTED;
    if (workspace != nullptr && !aligned16(workspace)) return LA_ERR_INVALID;
    if (!aligned16(state_pool) || (T > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) ||
                                             !aligned16(out))))
        return LA_ERR_INVALID;
    if (!aligned4(slopes) || !aligned4(state_idx) || !aligned4(cu_seqlens) ||
        (track_lens && (!aligned4(track_lens) || !aligned4(track_state_idx))))
        return LA_ERR_INVALID;
    la_status st;
    la::ExtendParams p{};
    if ((st = error_word_ptr(&p.err)) != LA_OK) return st;
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    p.k = reinterpret_cast<const __nv_bfloat16 *>(k);
    p.v = reinterpret_cast<const __nv_bfloat16 *>(v);
    p.slopes = slopes;
    p.pool = state_pool;
    p.state_idx = state_idx;
    p.cu_seqlens = cu_seqlens;
    p.prefix_mask = prefix_mask;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.B = B;
    p.T = T;
    p.H = H;
    p.Hkv = Hkv;
    p.group = H / Hkv;
    p.num_slots = num_slots;
    p.max_seqlen = max_seqlen;
    const unsigned long long us = g_wait_limit.load();
    p.wait_limit_ns = (us == 0 ? kDefaultWaitLimitUs : us) * 1000ull;
    p.seg_len = 0;
    p.blk_len = 0;
    p.nseg = 1;
    p.nblk = 0;
    p.ws = nullptr;
    p.lpt = (B > 1 && B <= kInCtaRankedRequests) ? 1 : 0;
    p.order = nullptr;
    p.track_lens = track_lens;
    p.track_idx = track_state_idx;
    p.out_rs = out_rs;
    p.out_hs = out_hs;
    ExtendScratch scr;
    if ((st = extend_scratch(B, T, H, Hkv, max_seqlen, &scr)) != LA_OK) return st;
    // a grouped call cannot run without its initial-state copies
    if (p.group > 1 && (workspace == nullptr || (unsigned long long)workspace_bytes < scr.copies))
        return LA_ERR_INVALID;
    if (p.group > 1) p.ws = static_cast<float *>(workspace);
    if (workspace != nullptr && scr.plan.seg_len > 0 &&
        (unsigned long long)workspace_bytes >= scr.full) {
        p.seg_len = scr.plan.seg_len;
        p.blk_len = scr.plan.blk_len;
        p.nseg = scr.plan.nseg;
        p.nblk = scr.plan.nblk;
        p.ws = static_cast<float *>(workspace);
    }
    // a large batch is taken longest first when the workspace has room for its order
    int32_t *order = nullptr;
    if (workspace != nullptr && scr.order > 0 &&
        (unsigned long long)workspace_bytes >= scr.full + scr.order) {
        order = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + scr.full);
        p.order = order;
        p.lpt = 1;
    }
    // Persistent grid: a batch of more (request, head) pairs than SMs runs on one CTA per SM
    // when the workspace has room for the request records.
    la::ItemRec *recs = nullptr;
    int many_ctas = 0;
    if (workspace != nullptr && scr.recs > 0 && g_persistent.load() &&
        (unsigned long long)workspace_bytes >= scr.full + scr.order + scr.recs) {
        int sms = 0;
        if ((st = num_sms(&sms)) != LA_OK) return st;
        recs = reinterpret_cast<la::ItemRec *>(static_cast<char *>(workspace) + scr.full +
                                               scr.order);
        many_ctas = sms;
    }
    // Column split: SMs that one CTA per (request, head) leaves idle take the second value-column
    // half of the longest requests, H CTAs per request.
    p.csplit = 0;
    if (p.seg_len == 0 && T > 0 && g_column_split.load() && (B == 1 || p.lpt)) {
        int sms = 0;
        if ((st = num_sms(&sms)) != LA_OK) return st;
        const long long spare = (long long)sms - (long long)B * H;
        if (spare >= H) p.csplit = (int)std::min<long long>(B, spare / H);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    p.recs = nullptr;
    // Balanced grid: a one-wave batch whose requests differ in length runs as segments planned
    // on the device, on one CTA per SM, when the workspace has room for the plan.
    if (workspace != nullptr && scr.bal > 0 && g_balanced.load() && p.seg_len == 0 &&
        p.group == 1 && T > 0 &&
        (unsigned long long)workspace_bytes >= scr.full + scr.order + scr.recs + scr.bal) {
        int sms = 0;
        if ((st = num_sms(&sms)) != LA_OK) return st;
        void *plan = static_cast<char *>(workspace) + scr.full + scr.order + scr.recs;
        return launch_status(la::launch_extend_bal(p, plan, sms, s));
    }
    if (many_ctas > 0 && p.seg_len == 0 && p.csplit == 0 && p.group == 1)
        return launch_status(la::launch_extend_many(p, recs, many_ctas, s));
    if (order != nullptr && la::launch_rank_requests(cu_seqlens, B, order, s) != cudaSuccess)
        return LA_ERR_CUDA;
    if (p.seg_len > 0 || p.group > 1) {
        cudaError_t e = la::launch_block_states(p, s);
        if (e == cudaSuccess) e = la::launch_state_scan(p, s);
        if (e != cudaSuccess) return LA_ERR_CUDA;
    }
    return launch_status(la::launch_extend_wide(p, s));
}

}  // namespace

extern "C" {

la_status la_extend(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                    float *state_pool, int num_slots, const int32_t *state_idx,
                    const int32_t *cu_seqlens, const uint8_t *prefix_mask, la_bf16 *out, int B,
                    int T, int H, int D, int max_seqlen, void *workspace, size_t workspace_bytes,
                    la_stream stream) {
    return extend_impl(q, k, v, slopes, state_pool, num_slots, state_idx, cu_seqlens, prefix_mask,
                       nullptr, nullptr, out, 0, 0, B, T, H, H, D, max_seqlen, workspace,
                       workspace_bytes, stream);
}

la_status la_extend_gqa(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                        float *state_pool, int num_slots, const int32_t *state_idx,
                        const int32_t *cu_seqlens, const uint8_t *prefix_mask, la_bf16 *out,
                        int B, int T, int H, int Hkv, int D, int max_seqlen, void *workspace,
                        size_t workspace_bytes, la_stream stream) {
    return extend_impl(q, k, v, slopes, state_pool, num_slots, state_idx, cu_seqlens, prefix_mask,
                       nullptr, nullptr, out, 0, 0, B, T, H, Hkv, D, max_seqlen, workspace,
                       workspace_bytes, stream);
}

la_status la_extend_gqa_workspace_size(int B, int T, int H, int Hkv, int D, int max_seqlen,
                                       size_t *bytes) {
    if (B < 0 || T < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || D < 1 || max_seqlen < 0 ||
        bytes == nullptr)
        return LA_ERR_INVALID;
    if (D != la::kHeadDim) return LA_ERR_UNSUPPORTED;
    ExtendScratch scr;
    const la_status st = extend_scratch(B, T, H, Hkv, max_seqlen, &scr);
    if (st != LA_OK) return st;
    *bytes = (size_t)(scr.full + scr.order + scr.recs + scr.bal);
    return LA_OK;
}

la_status la_decode_gqa(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                        float *state_pool, int num_slots, const int32_t *state_idx, la_bf16 *out,
                        int B, int H, int Hkv, int D, la_stream stream) {
    if (B < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || D < 1 || num_slots < 1)
        return LA_ERR_INVALID;
    if (D != la::kHeadDim) return LA_ERR_UNSUPPORTED;
    if (Hkv == H)  // one query head per state: the plain decode
        return la_decode(q, k, v, slopes, state_pool, num_slots, state_idx, out, B, H, D, stream);
    if (B == 0) return LA_OK;
    if (!q || !k || !v || !slopes || !state_pool || !state_idx || !out) return LA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state_pool) ||
        !aligned16(out) || !aligned4(slopes) || !aligned4(state_idx))
        return LA_ERR_INVALID;
    la::RecurParams p{};
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    p.k = reinterpret_cast<const __nv_bfloat16 *>(k);
    p.v = reinterpret_cast<const __nv_bfloat16 *>(v);
    p.slopes = slopes;
    p.pool = state_pool;
    p.state_idx = state_idx;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.B = B;
    p.H = Hkv;
    p.G = H / Hkv;
    p.N = 1;
    p.num_slots = num_slots;
    la_status st = error_word_ptr(&p.err);
    if (st != LA_OK) return st;
    return launch_status(la::launch_decode_grouped(p, static_cast<cudaStream_t>(stream)));
}

la_status la_extend_ex(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                       float *state_pool, int num_slots, const int32_t *state_idx,
                       const int32_t *cu_seqlens, const uint8_t *prefix_mask,
                       const int32_t *track_lens, const int32_t *track_state_idx, la_bf16 *out,
                       int64_t out_row_stride, int64_t out_head_stride, int B, int T, int H, int D,
                       int max_seqlen, void *workspace, size_t workspace_bytes, la_stream stream) {
    if ((track_lens == nullptr) != (track_state_idx == nullptr)) return LA_ERR_INVALID;
    return extend_impl(q, k, v, slopes, state_pool, num_slots, state_idx, cu_seqlens, prefix_mask,
                       track_lens, track_state_idx, out, (long long)out_row_stride,
                       (long long)out_head_stride, B, T, H, H, D, max_seqlen, workspace,
                       workspace_bytes, stream);
}

la_status la_extend_workspace_size(int B, int T, int H, int D, int max_seqlen, size_t *bytes) {
    if (B < 0 || T < 0 || H < 1 || D < 1 || max_seqlen < 0 || bytes == nullptr)
        return LA_ERR_INVALID;
    if (D != la::kHeadDim) return LA_ERR_UNSUPPORTED;
    ExtendScratch scr;
    const la_status st = extend_scratch(B, T, H, H, max_seqlen, &scr);
    if (st != LA_OK) return st;
    *bytes = (size_t)(scr.full + scr.order + scr.recs + scr.bal);
    return LA_OK;
}

}  // extern "C"
