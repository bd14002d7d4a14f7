// la_extend_seg.cu -- sequence split of long extend requests: the split planner and the
// block-state kernel.
//
// Method: page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section
// "独立参考实现：逐 token 递推公式": S_t = S_{t-1} e^{-s} + outer(k_t, v_t).  Unrolled over a block
// of tokens [a, e) starting from zero, the state at the block's end is
//     B = sum_{t in [a, e)} e^{-s (e - 1 - t)} outer(k_t, v_t),
// and the state at any later token boundary x is e^{-s (x - e)} B plus the contributions of the
// tokens after e.  So a request can be cut into segments processed in parallel: segment g starts
// from e^{-s x_g} S0 + sum over the blocks k before x_g of e^{-s (x_g - e_k)} B_k (positions
// relative to the request's first token).  That is a reassociation of the same sum, exact up to
// rounding.
//
// The block-state kernel computes B_k for the blocks that precede a request's last segment, and
// copies each split request's initial state S0 (its pool slot, or zero) into the workspace, so
// that the extend kernel's segments never read a pool slot that the last segment rewrites.  For a
// grouped-query call (several query heads per kv head) it copies every request's S0, for the same
// reason: the group's first query head rewrites the slot that its siblings start from.
//
// One CTA per (request, head, block): a TMA warp streams the block's K and V tiles (C x 128 each,
// three stages), last chunk first: the extend kernel starts each segment at its first chunk, so
// the tiles read last here are the first it reads again, while some are still in L2 (the terms
// of B do not depend on the order they are summed in).  Eight warps scale K by e^{-s (e - 1 - t)}
// into a bf16 pair hi (in place) + lo; one thread issues tcgen05.mma (bf16 x bf16 -> fp32)
// accumulating B = K_hi^T V + K_lo^T V in tensor memory over the whole block, V straight from the
// TMA tile; the eight warps then write B (fp32, 64 KiB) to the workspace.  The decay factors of a block span its whole length, so one
// 16-bit K_hat would round every term by up to 2^-9 (bf16) or 2^-11 (fp16), an error that the
// state of a slowly decaying head sums over thousands of tokens; the pair keeps the terms to
// about 2^-17.  The work is HBM bound (64 KiB of K and V per 128 tokens, 4 x 128 x 128 x 128 MMA
// flops).
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {

namespace {

using namespace sm100;

constexpr int C = 128;
constexpr int kConvWarps = 8;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t SZ_T = C * kHeadDim * 2;   // one [C][128] 16-bit tile: two 16 KiB blocks
constexpr uint32_t SZ_STAGE = 2 * SZ_T;       // K (lambda K hi after conversion) and V of a chunk
constexpr int kStages = 3;                    // three chunks in flight hide the load latency
constexpr uint32_t OFF_KLO = kStages * SZ_STAGE;  // lambda K lo of the chunk being multiplied
constexpr uint32_t OFF_BAR = OFF_KLO + SZ_T;
constexpr uint32_t kSmemBytes = OFF_BAR + 128 + 1024;
static_assert(SZ_STAGE % 1024 == 0, "atoms");

struct Bars {
    uint64_t full[kStages];   // TMA -> converters
    uint64_t conv[kStages];   // converters -> MMA (8 warp arrivals)
    uint64_t empty[kStages];  // MMA -> TMA
    uint64_t done;      // every MMA of the block completed
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= 128, "barrier block");
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint64_t kDrainLimitNs = 2000000000ull;

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                         volatile int *abort_flag, unsigned int *err) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(a, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicOr(err, ERR_BIT_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int *abort_flag, unsigned int *err) {
    const bool ok = wait_bar(bar, parity, limit_ns, abort_flag, err);
    return __all_sync(0xffffffffu, ok);
}

__global__ void __launch_bounds__(kThreads, 1)
    block_state_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                       const ExtendParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw);
    Bars *bars = reinterpret_cast<Bars *>(sm + OFF_BAR);
    pdl_wait();
    pdl_trigger();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = p.Hkv;  // the states' heads (kv heads of a grouped call)
    const int nblk_grid = p.nblk > 0 ? p.nblk : 1;
    const int k = blockIdx.x % nblk_grid;
    const int bh = blockIdx.x / nblk_grid;
    const int h = bh % H;
    const int b = bh / H;

    const int slot = p.state_idx[b];
    const int t0 = p.cu_seqlens[b];
    const int t1 = p.cu_seqlens[b + 1];
    if (slot < 0 || slot >= p.num_slots || t0 < 0 || t1 < t0 || t1 > p.T) return;  // the extend
    // kernel, launched next on the same stream, records these faults in the error word
    const int n = t1 - t0;
    if (n > p.max_seqlen) return;  // longer than the caller's bound: reported by the extend kernel
    const int nseg_b = p.seg_len > 0 ? (n + p.seg_len - 1) / p.seg_len : 1;
    if (nseg_b <= 1 && p.group == 1) return;  // not split: nothing to copy or compute
    float *ws_bh = p.ws + ((size_t)b * H + h) * (size_t)(1 + p.nblk) * (kHeadDim * kHeadDim);

    // The initial state S0 of a split request (pool slot if it has a prefix, else zero).
    if (k == 0 && threadIdx.x < kConvThreads) {
        const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
        const float *src =
            p.pool + (((size_t)slot * H + h) * kHeadDim + row) * kHeadDim + half * 64;
        float *dst = ws_bh + (size_t)row * kHeadDim + half * 64;
        const bool pre = p.prefix_mask[b] != 0;
#pragma unroll
        for (int x = 0; x < 16; ++x)
            reinterpret_cast<float4 *>(dst)[x] =
                pre ? reinterpret_cast<const float4 *>(src)[x] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (nseg_b <= 1) return;  // grouped call, request not split: the copy was all
    const int per_seg = p.seg_len / p.blk_len;
    if (k >= (nseg_b - 1) * per_seg) return;  // block at or after the last segment's start

    const int a = k * p.blk_len;               // block [a, e) relative to t0; always full length
    const int nchunks = p.blk_len / C;
    const uint64_t limit = p.wait_limit_ns;
    const float slope = p.slopes[h];

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->conv[s], kConvWarps);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->done, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bars->tmem_base;
    volatile int *abort_flag = &bars->abort_flag;
    const uint32_t s_base = smem_u32(sm);

    if (warp == kProducerWarp) {
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % kStages;
                if (c >= kStages && !wait_bar(&bars->empty[st], (c / kStages - 1) & 1, limit,
                                              abort_flag, p.err))
                    break;
                const int y = t0 + a + (nchunks - 1 - c) * C;  // last chunk first
                const int x = h * kHeadDim;
                uint8_t *dst = sm + st * SZ_STAGE;
                mbar_arrive_expect_tx(&bars->full[st], SZ_STAGE);
                tma_load_2d(dst, &tk, &bars->full[st], x, y);
                tma_load_2d(dst + 16384, &tk, &bars->full[st], x + 64, y);
                tma_load_2d(dst + SZ_T, &tv, &bars->full[st], x, y);
                tma_load_2d(dst + SZ_T + 16384, &tv, &bars->full[st], x + 64, y);
                issued = c + 1;
            }
            for (int c = (issued >= kStages ? issued - kStages : 0); c < issued; ++c) {
                int dummy = 0;
                wait_bar(&bars->full[c % kStages], (c / kStages) & 1, kDrainLimitNs, &dummy,
                         p.err);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // one N = 128 MMA per 16 tokens: an M = 128 instruction costs about the same at
            // N = 64 as at N = 128
            const uint32_t idU = idesc_bf16_f32(128, 128, true, true);
            const uint64_t dK0 = sdesc_sw128(s_base, 16384, 1024);         // K^T: MN-major A
            const uint64_t dV0 = sdesc_sw128(s_base + SZ_T, 16384, 1024);  // V: MN-major B
            const uint64_t dKlo = sdesc_sw128(s_base + OFF_KLO, 16384, 1024);
            const uint64_t step = SZ_STAGE >> 4;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % kStages;
                if (!wait_bar(&bars->conv[st], (c / kStages) & 1, limit, abort_flag, p.err))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase, dK0 + st * step + (uint64_t)(kk * 128),
                             dV0 + st * step + (uint64_t)(kk * 128), idU,
                             (c > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase, dKlo + (uint64_t)(kk * 128),
                             dV0 + st * step + (uint64_t)(kk * 128), idU, 1u);
                mma_commit(&bars->empty[st]);
            }
            mma_commit(&bars->done);
            int dummy = 0;
            wait_bar(&bars->done, 0, kDrainLimitNs, &dummy, p.err);
        }
    } else {
        // converters / epilogue: thread pair (2 row, 2 row + 1) owns row `row` of the chunk; each
        // scales one 64-column half of K
        const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
            const int st = c % kStages;
            if (!(ok = warp_wait_bar(&bars->full[st], (c / kStages) & 1, limit, abort_flag,
                                     p.err)))
                break;
            // distance of this token to the block's last token: (blk_len - 1) - (cc C + row), where
            // cc = nchunks - 1 - c is the chunk's place in the block
            const int cc = nchunks - 1 - c;
            const LamSplitBf lam =
                lam_split_bf16(expf(-slope * (float)(p.blk_len - 1 - cc * C - row)));
            uint4 *krow = reinterpret_cast<uint4 *>(sm + st * SZ_STAGE + half * 16384 + row * 128);
            uint4 *lrow = reinterpret_cast<uint4 *>(sm + OFF_KLO + half * 16384 + row * 128);
            const int rot = row + half * 4;  // 8 threads of a quarter-warp hit 8 distinct banks
            uint4 kb[8];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) kb[ch] = krow[(ch + rot) & 7];
            uint4 lo[8];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint4 hi;
                bf16x8_lam_hilo_bf16(kb[ch], lam, hi, lo[ch]);
                krow[(ch + rot) & 7] = hi;
            }
            // the lo buffer is free once the MMAs of the previous chunk are done with it
            if (c >= 1) {
                const int prev = (c - 1) % kStages;
                if (!(ok = warp_wait_bar(&bars->empty[prev], ((c - 1) / kStages) & 1, limit,
                                         abort_flag, p.err)))
                    break;
            }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) lrow[(ch + rot) & 7] = lo[ch];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->conv[st]);
        }
        if (ok && warp_wait_bar(&bars->done, 0, limit, abort_flag, p.err)) {
            tc_fence_after();
            const int q = warp & 3, wg = warp >> 2;
            const int i = q * 32 + lane;
            float *dst = ws_bh + (size_t)(1 + k) * (kHeadDim * kHeadDim) + (size_t)i * kHeadDim +
                         wg * 64;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t v[32];
                tmem_ld32(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(wg * 64 + hh * 32), v);
                tmem_ld_wait_regs(v);
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    reinterpret_cast<float4 *>(dst + hh * 32)[x] =
                        make_float4(__uint_as_float(v[4 * x]), __uint_as_float(v[4 * x + 1]),
                                    __uint_as_float(v[4 * x + 2]), __uint_as_float(v[4 * x + 3]));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// Segment start states from the block states, in place.  With T_{-1} = S0 and every block of
// blk_len tokens, T_k = e^{-s blk_len} T_{k-1} + B_k is the state after block k (the same sum the
// segments would otherwise form term by term), and segment g starts from T_{g P - 1}, P blocks per
// segment; the kernel overwrites block state g P - 1 with it, so that a segment's prologue reads
// one matrix however far into the request it starts.  Four CTAs of 1024 threads per (request,
// head), one float4 of the 128 x 128 state per thread: the scan is elementwise, and each thread
// keeps eight block states' loads in flight ahead of its multiply-adds, so the serial chain over
// the blocks costs one L2 round trip per eight blocks.
constexpr int kScanThreads = 1024;
constexpr int kScanAhead = 8;

__global__ void __launch_bounds__(kScanThreads) state_scan_kernel(const ExtendParams p) {
    pdl_wait();
    pdl_trigger();
    const int H = p.Hkv;
    const int part = blockIdx.x & 3;
    const int bh = blockIdx.x >> 2;
    const int h = bh % H;
    const int b = bh / H;
    const int slot = p.state_idx[b];
    const int t0 = p.cu_seqlens[b];
    const int t1 = p.cu_seqlens[b + 1];
    if (slot < 0 || slot >= p.num_slots || t0 < 0 || t1 < t0 || t1 > p.T) return;  // reported by
    const int n = t1 - t0;                                                         // the extend
    if (n > p.max_seqlen) return;                                                   // kernel
    const int nseg_b = (n + p.seg_len - 1) / p.seg_len;
    if (nseg_b <= 1) return;
    const int per_seg = p.seg_len / p.blk_len;
    const int nk = (nseg_b - 1) * per_seg;  // blocks before the last segment
    constexpr int kVec = kHeadDim * kHeadDim / 4;  // float4 per state
    float4 *ws = reinterpret_cast<float4 *>(p.ws + ((size_t)b * H + h) * (size_t)(1 + p.nblk) *
                                                       (kHeadDim * kHeadDim));
    const int e = part * kScanThreads + threadIdx.x;
    const float d = expf(-p.slopes[h] * (float)p.blk_len);
    float4 t = __ldcg(ws + e);  // S0
    for (int k0 = 0; k0 < nk; k0 += kScanAhead) {
        float4 bk[kScanAhead];
#pragma unroll
        for (int j = 0; j < kScanAhead; ++j)
            if (k0 + j < nk) bk[j] = __ldcg(ws + (size_t)(1 + k0 + j) * kVec + e);
#pragma unroll
        for (int j = 0; j < kScanAhead; ++j) {
            const int k = k0 + j;
            if (k < nk) {
                t.x = fmaf(d, t.x, bk[j].x);
                t.y = fmaf(d, t.y, bk[j].y);
                t.z = fmaf(d, t.z, bk[j].z);
                t.w = fmaf(d, t.w, bk[j].w);
                if ((k + 1) % per_seg == 0) ws[(size_t)(1 + k) * kVec + e] = t;
            }
        }
    }
}

}  // namespace

// Split only when the batch leaves SMs idle: with u = B * H * 2 extend CTAs (two v blocks per
// head) and u < num_sms / 2, cut each request into G = floor(num_sms / u) segments (at least
// 8 chunks each), and each segment into P blocks so that the block-state kernel also fills the
// GPU.  Workspace: B * H * (1 + nblk) fp32 D x D matrices.
SplitPlan plan_split(int B, int H, int max_seqlen, int num_sms, int ctas_per_head) {
    SplitPlan pl{0, 0, 1, 0, 0ull};
    const long long units = (long long)B * H * ctas_per_head;
    if (B <= 0 || units <= 0 || num_sms <= 0 || 2 * units > num_sms) return pl;
    const int min_seg = 8 * C;
    int G = (int)(num_sms / units);
    const int by_len = max_seqlen / min_seg;
    if (by_len < G) G = by_len;
    if (G < 2) return pl;
    const int seg0 = (max_seqlen + G - 1) / G;
    const long long bh = (long long)B * H;
    int P = (int)(num_sms / (bh * (G - 1)));
    const int p_len = (seg0 + min_seg - 1) / min_seg;
    if (P > p_len) P = p_len;
    if (P < 1) P = 1;
    const int blk = ((seg0 + P - 1) / P + C - 1) / C * C;
    pl.blk_len = blk;
    pl.seg_len = blk * P;
    pl.nseg = (max_seqlen + pl.seg_len - 1) / pl.seg_len;
    if (pl.nseg < 2) return SplitPlan{0, 0, 1, 0, 0ull};
    pl.nblk = (pl.nseg - 1) * P;
    pl.ws_bytes = (unsigned long long)bh * (unsigned long long)(1 + pl.nblk) * kHeadDim * kHeadDim *
                  sizeof(float);
    return pl;
}


namespace {

// order[rank of b] = b, ranks by decreasing length (request_rank).
__global__ void __launch_bounds__(256) rank_requests_kernel(const int32_t *cu_seqlens, int B,
                                                            int32_t *order) {
    pdl_wait();
    pdl_trigger();
    __shared__ int lens[256];
    const int b = blockIdx.x * 256 + threadIdx.x;
    const int lb = b < B ? cu_seqlens[b + 1] - cu_seqlens[b] : 0;
    const int rank = request_rank(cu_seqlens, B, b, lb, lens);
    if (b < B) order[rank] = b;
}

}  // namespace

cudaError_t launch_rank_requests(const int32_t *cu_seqlens, int B, int32_t *order,
                                 cudaStream_t stream) {
    if (B <= 0) return cudaSuccess;
    return launch_pdl(rank_requests_kernel, dim3((unsigned)((B + 255) / 256)), dim3(256), 0, stream,
                      cu_seqlens, B, order);
}

cudaError_t launch_state_scan(const ExtendParams &p, cudaStream_t stream) {
    if (p.seg_len <= 0 || p.nblk <= 0) return cudaSuccess;
    const long long ctas = (long long)p.B * p.Hkv * 4;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_pdl(state_scan_kernel, dim3((unsigned)ctas), dim3(kScanThreads), 0, stream, p);
}

cudaError_t launch_block_states(const ExtendParams &p, cudaStream_t stream) {
    if (p.seg_len <= 0 && p.group == 1) return cudaSuccess;
    const long long ctas = (long long)p.B * p.Hkv * (p.nblk > 0 ? p.nblk : 1);
    if (ctas <= 0) return cudaSuccess;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap tk, tv;
    memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv));
    if (p.T > 0 && (!make_token_map_full(&tk, p.k, p.T, p.Hkv) ||
                    !make_token_map_full(&tv, p.v, p.T, p.Hkv)))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static bool configured[64] = {false};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!configured[dev]) {
            e = cudaFuncSetAttribute(block_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBytes);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    return launch_pdl(block_state_kernel, dim3((unsigned)ctas), dim3(kThreads), kSmemBytes, stream,
                      tk, tv, p);
}

}  // namespace la
