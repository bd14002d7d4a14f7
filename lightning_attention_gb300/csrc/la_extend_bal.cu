// la_extend_bal.cu -- chunked seg_la extend for batches that fit in one wave but whose requests
// differ in length: a planner cuts the longest requests into segments so that every SM gets about
// the same work, and a persistent grid of one CTA per SM runs the segments.
//
// Method: page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section
// "独立参考实现：逐 token 递推公式" (per head, S_t = S_{t-1} e^{-s} + outer(k_t, v_t) and
// o_t = (q_t @ S_t) D^-0.5 from the request's pool state or zero, final state written back), in
// the chunked form that la_extend_w.cu states; state-tracking snapshots as in section "额外覆盖".
// A segment [a, e) of a request starts from the state after its first a tokens,
//     S_a = e^{-s a} S0 + sum_{t < a} e^{-s (a - 1 - t)} outer(k_t, v_t),
// which is the same sum regrouped (exact up to rounding).  The segment's CTA forms S_a itself:
// a prologue over the request's first a tokens, in chunks of C, that only scales K by those
// factors (as a bf16 pair hi + lo, like the state update) and accumulates (lambda K)^T V onto
// e^{-s a} S0 in tensor memory.  It reads the K and V of those tokens a second time, but it waits
// for no other CTA's result.
//
// Why.  One CTA per (request, head) keeps B H SMs busy and lasts as long as the longest request;
// in a batch of uneven lengths most SMs finish early and idle (8 requests of 5 to 30 chunks on 16
// heads: 128 CTAs, the kernel ends with the 30-chunk request while the mean is 16 chunks per SM).
// Cutting the long requests evens out the load at the price of the prologue's reads.
//
// Plan (seg_plan_kernel, one block).  Costs are counted in tenths of a chunk, as measured with every
// SM streaming: 10 per chunk of a segment, 5 per prologue chunk (half a chunk's bytes), 12 per item
// (loading its start state, writing its final state).
// For a target item cost M, a request of n chunks is cut from its start: each segment takes as
// many chunks as keep its cost within M, at least two, and a remainder shorter than two chunks
// joins the segment before it.  Sixteen targets from the mean load per CTA up to the longest
// request (no cut) are tried on those cuts, one per warp.  For each, the segments' items (one per head) are put
// in order -- the non-last segments of cut requests first, then the rest, each by decreasing cost
// -- and dealt to the P CTAs in snake order (CTA j takes ranks j, 2P - 1 - j, 2P + j, ...); the
// target with the smallest largest CTA load wins (ties: fewer segments).  Its requests are then cut
// into as many segments as before with the smallest target that needs no more, which evens out
// their costs and shortens the first segments, whose keys and values the later ones read again.  Targets that need more
// than 2P items, or more than P items of non-last segments, are not taken.
//
// The initial state of a cut request.  Each segment of a request with a prefix reads S0 from the
// request's pool slot, which the last segment overwrites with the final state.  The non-last
// segments are dealt first, so each is the first item of its CTA; after reading S0 each of its
// epilogue warps adds one to a counter of the (request, head), and the last segment's warps wait
// (bounded) for all of those counts before they write the slot.  The first items wait for nothing
// before their read, so that wait ends.
//
// Per chunk the roles, buffers, barriers and orders are those of la_extend_w.cu and
// la_extend_many.cu.  A prologue chunk loads no Q, so two of them are in flight: their V goes
// alternately into the V and the (idle) Q buffer, their lambda K lo alternately into its buffer
// and S_hi's (idle until the prologue ends), with a barrier pair per lo buffer (kp_ready: lambda K
// written; pro_done: the chunk's MMAs done).  The K ring's barriers count every chunk of the CTA's
// stream, the Q and V buffers' barriers count their uses, the A, K-ready, P, U and O barriers
// count the segments' own chunks, and s_ready completes once more per item with a prologue (its
// seed, then the pass that turns S_a into the first chunk's operands).  No barrier can complete
// twice before its waiter has seen the first completion, so every parity wait is unambiguous.
#include <string.h>

#include <mutex>

#include "la_extend_bal.h"
#include "la_extend_tile.cuh"

namespace la {

namespace {

constexpr int kPlanWarps = 16;              // targets tried, one per warp
constexpr int kPlanThreads = kPlanWarps * 32;
constexpr int kCostChunk = 10;              // cost of one chunk of a segment (tenths of a chunk)
constexpr int kCostPro = 5;                 // of one prologue chunk
constexpr int kCostItem = 12;               // of starting and ending an item
constexpr int kMinSegChunks = 2;            // shortest segment of a cut request, in chunks
constexpr int kMaxSegs = 8;                 // segments of one request

// Greedy cut of a request of nc > 0 chunks for target cost M: each segment takes the chunks that
// keep its cost within M (at least kMinSegChunks; a shorter remainder joins it).  Writes the
// segment ends (in chunks) when `ends` is given; returns the count.
__device__ __forceinline__ int cut_greedy(int nc, int M, int *ends) {
    int a = 0, m = 0;
    while (a < nc) {
        int l = (M - kCostItem - kCostPro * a) / kCostChunk;
        if (l < kMinSegChunks) l = kMinSegChunks;
        int e = a + l;
        if (e >= nc || nc - e < kMinSegChunks || m == kMaxSegs - 1) e = nc;
        if (ends != nullptr) ends[m] = e;
        ++m;
        a = e;
    }
    return m;
}

// Cut a request of nc chunks for target cost M: as many segments as the greedy cut makes, with the
// smallest target that still needs no more, so that the segments' costs come out about equal (and
// the first ones, whose keys and values the later ones read again, no longer than they must).
// Returns the count (one segment of no chunks for an empty request).
__device__ __forceinline__ int cut_request(int nc, int M, int (&ends)[kMaxSegs]) {
    if (nc <= 0) {
        ends[0] = 0;
        return 1;
    }
    const int m = cut_greedy(nc, M, nullptr);
    if (m > 1) {
        // m segments cover nc chunks, so one of them costs at least nc / m chunks and an item
        int lo = kCostChunk * (nc / m) + kCostItem, hi = M;  // cut_greedy(nc, hi) <= m throughout
        if (lo > hi) lo = hi;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (cut_greedy(nc, mid, nullptr) <= m) hi = mid;
            else lo = mid + 1;
        }
        M = hi;
    }
    return cut_greedy(nc, M, ends);
}

__device__ __forceinline__ int seg_cost(int a, int e) {
    return kCostChunk * (e - a) + kCostPro * a + kCostItem;
}

// Sort key: non-last segments of cut requests first, then by decreasing cost.
__device__ __forceinline__ int seg_key(int cost, bool nonlast) {
    return cost + (nonlast ? (1 << 24) : 0);
}

// The request facts the plan needs, staged in shared memory by the validation step.
struct PlanReq {
    int nc;      // chunks (-1: faulty request, skipped)
    int t0, n, slot, tl, tslot, prefix;
};

// Plan: validate the requests (reporting faults as the other extend kernels do), choose the
// target, write the records in deal order and zero the read counters.
__global__ void __launch_bounds__(kPlanThreads) seg_plan_kernel(const ExtendParams p, int P,
                                                                SegHeader *hdr, SegRec *recs,
                                                                int *counters) {
    pdl_wait();
    pdl_trigger();
    __shared__ PlanReq req[kMaxBalRequests];
    __shared__ int s_key[kPlanWarps][kMaxBalRecs];
    __shared__ int s_sorted[kPlanWarps][kMaxBalRecs];
    __shared__ int s_rb[kMaxBalRecs], s_ra[kMaxBalRecs], s_re[kMaxBalRecs], s_rm[kMaxBalRecs];
    __shared__ int s_span[kPlanWarps];
    __shared__ int s_M[kPlanWarps];
    __shared__ int s_best;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = p.B, H = p.H;

    for (int b = threadIdx.x; b < B; b += kPlanThreads) {
        PlanReq r{-1, 0, 0, 0, -1, 0, 0};
        // every load first (they are independent), then the checks
        const int t0 = p.cu_seqlens[b], t1 = p.cu_seqlens[b + 1];
        const int slot = p.state_idx[b];
        const int pre = p.prefix_mask[b];
        const int tl = p.track_lens != nullptr ? p.track_lens[b] : -1;
        const int ts = p.track_lens != nullptr ? p.track_idx[b] : 0;
        const int n = t1 - t0;
        if (slot < 0 || slot >= p.num_slots) {
            atomicOr(p.err, ERR_BIT_SLOT_RANGE);
        } else if (t0 < 0 || t1 < t0 || t1 > p.T || n > p.max_seqlen) {
            atomicOr(p.err, ERR_BIT_SEQLENS);
        } else {
            r = PlanReq{(n + C - 1) / C, t0, n, slot, -1, 0, pre ? 1 : 0};
            {
                if (tl >= 0) {
                    if (tl > n || ts < 0 || ts >= p.num_slots || ts == slot) {
                        atomicOr(p.err, ERR_BIT_TRACK);
                    } else {
                        r.tl = tl;
                        r.tslot = ts;
                    }
                }
            }
        }
        req[b] = r;
    }
    for (int x = threadIdx.x; x < B * H; x += kPlanThreads) counters[x] = 0;
    __syncthreads();

    // The range of targets: from the mean load per CTA to the longest request uncut.
    int tot = 0, mx = 0;
    for (int b = lane; b < B; b += 32) {
        const int nc = req[b].nc;
        if (nc >= 0) {
            tot += seg_cost(0, nc);
            mx = max(mx, seg_cost(0, nc));
        }
    }
    tot = __reduce_add_sync(0xffffffffu, tot);
    mx = __reduce_max_sync(0xffffffffu, mx);
    const int lo = min(mx, max(seg_cost(0, kMinSegChunks),
                               (int)(((long long)tot * H + P - 1) / P)));
    const int M = lo + (int)((long long)(mx - lo) * warp / (kPlanWarps - 1));

    // This warp's target: cut, order, deal, and measure the largest CTA load.
    int R = 0, nonlast = 0;
    bool ok = true;
    for (int b0 = 0; b0 < B; b0 += 32) {
        const int b = b0 + lane;
        int ends[kMaxSegs];
        int m = 0;
        // the targets are compared on their greedy cuts (the equalised cut of the chosen one
        // below costs no more); an empty request is one segment of no chunks
        const int nc = b < B ? req[b].nc : -1;
        if (nc > 0) {
            m = cut_greedy(nc, M, ends);
        } else if (nc == 0) {
            ends[0] = 0;
            m = 1;
        }
        int off = m;  // inclusive scan of the segment counts
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, off, d);
            if (lane >= d) off += y;
        }
        const int total = __shfl_sync(0xffffffffu, off, 31);
        off -= m;
        if (R + total > kMaxBalRecs) {
            ok = false;
            break;
        }
        int a = 0;
        for (int s = 0; s < m; ++s) {
            s_key[warp][R + off + s] = seg_key(seg_cost(a, ends[s]), s + 1 < m);
            a = ends[s];
        }
        nonlast += __reduce_add_sync(0xffffffffu, m > 1 ? m - 1 : 0);
        R += total;
    }
    if (ok && ((long long)R * H > 2ll * P || (long long)nonlast * H > P)) ok = false;
    __syncwarp();
    int span = 0x7fffffff;
    if (ok) {
        // rank by key, ties by index: a permutation
        for (int x = lane; x < R; x += 32) {
            const int kx = s_key[warp][x];
            int rank = 0;
            for (int y = 0; y < R; ++y) {
                const int ky = s_key[warp][y];
                rank += (ky > kx) || (ky == kx && y < x);
            }
            s_sorted[warp][rank] = kx & ((1 << 24) - 1);
        }
        __syncwarp();
        int worst = 0;
        // at most 2P items (checked above): two rows of the deal; record of rank rk is rk / H
        const int items = R * H;
        for (int j = lane; j < P; j += 32) {
            int load = j < items ? s_sorted[warp][j / H] : 0;
            const int rk = 2 * P - 1 - j;
            if (rk < items) load += s_sorted[warp][rk / H];
            worst = max(worst, load);
        }
        span = __reduce_max_sync(0xffffffffu, worst);
    }
    if (lane == 0) {
        s_span[warp] = span;
        s_M[warp] = M;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int best = kPlanWarps - 1;  // the largest target: never refused
        for (int w = kPlanWarps - 2; w >= 0; --w)
            if (s_span[w] < s_span[best]) best = w;
        s_best = best;
    }
    __syncthreads();

    // The chosen target's records, written at their rank (warp 0; the other warps are done).
    // Each lane cuts its own requests once; the records' requests and bounds go to shared memory.
    if (warp != 0) return;
    const int Mb = s_M[s_best];
    R = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
        const int b = b0 + lane;
        int ends[kMaxSegs];
        int m = 0;
        if (b < B && req[b].nc >= 0) m = cut_request(req[b].nc, Mb, ends);
        int off = m;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, off, d);
            if (lane >= d) off += y;
        }
        const int total = __shfl_sync(0xffffffffu, off, 31);
        off -= m;
        int a = 0;
        for (int sg = 0; sg < m; ++sg) {
            const int x = R + off + sg;
            s_key[0][x] = seg_key(seg_cost(a, ends[sg]), sg + 1 < m);
            s_rb[x] = b;
            s_ra[x] = a;
            s_re[x] = ends[sg];
            s_rm[x] = m;
            a = ends[sg];
        }
        R += total;
    }
    __syncwarp();
    for (int x = lane; x < R; x += 32) {
        const int kx = s_key[0][x];
        int rank = 0;
        for (int y = 0; y < R; ++y) {
            const int ky = s_key[0][y];
            rank += (ky > kx) || (ky == kx && y < x);
        }
        const int b = s_rb[x], m = s_rm[x];
        const PlanReq &q = req[b];
        const int ta = s_ra[x] * C;              // segment start, request-local token
        const int te = min(s_re[x] * C, q.n);    // segment end
        const int len = te - ta;
        const bool last = te == q.n;
        // the snapshot belongs to the segment holding the tracked token (the last one when it
        // is the request's end); sp is relative to the segment, len + 1: none
        int sp = len + 1;
        if (q.tl >= 0 && ((q.tl >= ta && q.tl < te) || (q.tl == te && last))) sp = q.tl - ta;
        const int nchunks =
            sp <= len ? (sp + C - 1) / C + (len - sp + C - 1) / C : (len + C - 1) / C;
        const int flags = kRecValid | (q.prefix ? kRecPrefix : 0) | (last ? kRecLast : 0);
        int4 *dst = reinterpret_cast<int4 *>(recs + rank);
        dst[0] = make_int4(b, q.t0 + ta, len, q.slot);
        dst[1] = make_int4(sp, q.tslot, nchunks, flags);
        dst[2] = make_int4(ta, m, 0, 0);
    }
    if (lane == 0) {
        hdr->nrec = R;
        hdr->target = Mb;
    }
}

// One (segment, head) item of a CTA's stream.
struct SegItem {
    SegRec r;
    int h;
    __device__ bool prefix() const { return (r.flags & kRecPrefix) != 0; }
    __device__ bool last() const { return (r.flags & kRecLast) != 0; }
    __device__ int npro() const { return r.a / C; }
    // this segment's epilogue warps count their read of S0 (a cut request with a prefix)
    __device__ bool signals() const { return r.nseg > 1 && !last() && prefix(); }
};

__device__ __forceinline__ bool load_seg_item(const SegRec *recs, int nrec, int H, int k,
                                              SegItem &it) {
    const long long G = gridDim.x, j = blockIdx.x;
    const long long rk = (k & 1) ? (long long)(k + 1) * G - 1 - j : (long long)k * G + j;
    if (rk >= (long long)nrec * H) return false;
    const int4 *src = reinterpret_cast<const int4 *>(recs + rk / H);
    const int4 x = __ldg(src), y = __ldg(src + 1), z = __ldg(src + 2);
    it.r = SegRec{x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w, z.x, z.y, 0, 0};
    it.h = (int)(rk % H);
    return true;
}

// A role's walk over its CTA's items: take() moves to the next item that has chunks, handing the
// empty ones it passes to `finish`.
struct SegWalk {
    int k = 0;
    bool more = false;
    SegItem nxt;
    __device__ __forceinline__ void start(const SegRec *recs, int nrec, int H) {
        more = load_seg_item(recs, nrec, H, 0, nxt);
    }
    template <class Finish>
    __device__ __forceinline__ bool take(const SegRec *recs, int nrec, int H, SegItem &out,
                                         Finish finish) {
        while (more) {
            out = nxt;
            more = load_seg_item(recs, nrec, H, ++k, nxt);
            if (out.r.nchunks > 0) return true;
            finish(out);
        }
        return false;
    }
};

// Buffer use counts of a CTA's stream, kept alike by the producer and the MMA issuer: gk K loads
// (the K ring), nq uses of the Q buffer, nv uses of the V buffer, gp prologue chunks.  A chunk of
// a segment loads Q into the Q buffer and V into the V buffer; prologue chunk gp, which has no Q,
// loads V into the V buffer when gp is even and into the Q buffer when it is odd, so two prologue
// chunks are in flight.
struct Uses {
    int gk = 0, nq = 0, nv = 0, gp = 0;
};

// One 32 KiB tile of `map` at token row y, columns x .. x + 127, into `dst` (two 64-column boxes).
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap &map, uint64_t *bar,
                                          int x, int y) {
    mbar_arrive_expect_tx(bar, SZ_T);
    tma_load_2d(dst, &map, bar, x, y);
    tma_load_2d(dst + 16384, &map, bar, x + 64, y);
}

// The TMA producer's loads of a prologue chunk: K into the ring, V into the V or the Q buffer.
__device__ __forceinline__ bool produce_kv(Bars *bars, uint8_t *sm, const CUtensorMap &tk,
                                           const CUtensorMap &tv, Uses &u, int y, int x,
                                           uint64_t limit, volatile int *abort_flag,
                                           unsigned int *err, Issued &is) {
    const int st = u.gk & 1;
    if (u.gk >= 2 &&
        !wait_bar(&bars->k_empty[st], ((u.gk >> 1) - 1) & 1, limit, abort_flag, err))
        return false;
    load_tile(sm + OFF_K + st * SZ_T, tk, &bars->k_full[st], x, y);
    is.k = ++u.gk;
    if ((u.gp & 1) == 0) {
        if (u.nv >= 1 && !wait_bar(&bars->v_empty, (u.nv - 1) & 1, limit, abort_flag, err))
            return false;
        load_tile(sm + OFF_V, tv, &bars->v_full, x, y);
        is.v = ++u.nv;
    } else {
        if (u.nq >= 1 && !wait_bar(&bars->q_empty, (u.nq - 1) & 1, limit, abort_flag, err))
            return false;
        load_tile(sm + OFF_Q, tv, &bars->q_full, x, y);
        is.q = ++u.nq;
    }
    ++u.gp;
    return true;
}

// The loads of a segment's chunk: K into the ring, Q and V into their buffers.
__device__ __forceinline__ bool produce_qkv(Bars *bars, uint8_t *sm, const CUtensorMap &tq,
                                            const CUtensorMap &tk, const CUtensorMap &tv, Uses &u,
                                            int y, int x, uint64_t limit,
                                            volatile int *abort_flag, unsigned int *err,
                                            Issued &is) {
    const int st = u.gk & 1;
    if (u.gk >= 2 &&
        !wait_bar(&bars->k_empty[st], ((u.gk >> 1) - 1) & 1, limit, abort_flag, err))
        return false;
    load_tile(sm + OFF_K + st * SZ_T, tk, &bars->k_full[st], x, y);
    is.k = ++u.gk;
    if (u.nq >= 1 && !wait_bar(&bars->q_empty, (u.nq - 1) & 1, limit, abort_flag, err))
        return false;
    load_tile(sm + OFF_Q, tq, &bars->q_full, x, y);
    is.q = ++u.nq;
    if (u.nv >= 1 && !wait_bar(&bars->v_empty, (u.nv - 1) & 1, limit, abort_flag, err))
        return false;
    load_tile(sm + OFF_V, tv, &bars->v_full, x, y);
    is.v = ++u.nv;
    return true;
}

// Lambda K of a prologue chunk as a bf16 pair (hi in place, lo into its buffer): row j of the
// chunk is token a - dist - C + j of the request, so its factor is e^{-s (dist + C - 1 - j)},
// its decay up to the segment start a.
__device__ __forceinline__ void lamk_pro_pass(uint8_t *sm, int st, uint32_t lo_off, int ku0,
                                              int lane, float slope, int dist) {
    uint4 kbuf[kKUnits][4];
    uint4 *krow[kKUnits];
    uint4 *lrow[kKUnits];
    int rr[kKUnits], h4[kKUnits];
#pragma unroll
    for (int k = 0; k < kKUnits; ++k) {
        const int u = ku0 + k;
        rr[k] = (u >> 2) * 32 + lane;
        const uint32_t roff = (u & 2) * 8192 + rr[k] * 128;
        krow[k] = reinterpret_cast<uint4 *>(sm + OFF_K + st * SZ_T + roff);
        lrow[k] = reinterpret_cast<uint4 *>(sm + lo_off + roff);
        h4[k] = (u & 1) * 4;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) kbuf[k][ch] = krow[k][(h4[k] + ch + rr[k]) & 7];
    }
#pragma unroll
    for (int k = 0; k < kKUnits; ++k) {
        const LamSplitBf lam = lam_split_bf16(expf(-slope * (float)(dist + C - 1 - rr[k])));
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            uint4 hi, lo;
            bf16x8_lam_hilo_bf16(kbuf[k][ch], lam, hi, lo);
            krow[k][(h4[k] + ch + rr[k]) & 7] = hi;
            lrow[k][(h4[k] + ch + rr[k]) & 7] = lo;
        }
    }
}

// This thread's rows of an item's start: S0 (pool slot with a prefix, else zero), columns
// col_base .. col_base + 63.  Without a prologue, as in the persistent kernel: a snapshot at the
// segment's token 0, then the bf16 pair for the first MMA2 and e^{-s r0} S0 into TMEM, or, for an
// empty request without a prefix, its (zero) final state.  With a prologue: e^{-s a} S0 into
// TMEM, onto which the prologue accumulates.  A warp of a non-last segment of a cut request with a
// prefix then counts its read.
template <bool kEx>
__device__ __forceinline__ void seed_seg(const ExtendParams &p, const SegItem &it, uint32_t t_s,
                                         int col_base, uint8_t *s_hi, uint8_t *s_lo, int i,
                                         int lane, int *counters) {
    const SegRec &r = it.r;
    const int npro = it.npro();
    const bool snap0 = kEx && r.sp == 0 && npro == 0;
    if (r.nchunks == 0 && !snap0 && it.prefix()) return;  // the slot already holds the state
    const float slope = p.slopes[it.h];
    const int r0 = r.nchunks > 0 ? chunk_len(kEx, 0, r.sp, r.len) : 0;
    const float d0s = expf(-slope * (float)(npro > 0 ? r.a : r0));
    const float *src =
        p.pool + (((size_t)r.slot * p.H + it.h) * kHeadDim + i) * kHeadDim + (size_t)col_base;
#pragma unroll 1
    for (int sub = 0; sub < 2; ++sub) {
        const int col0 = col_base + sub * 32;
        float S[32];
        if (it.prefix()) {
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float4 f = *reinterpret_cast<const float4 *>(src + sub * 32 + 4 * x);
                S[4 * x] = f.x;
                S[4 * x + 1] = f.y;
                S[4 * x + 2] = f.z;
                S[4 * x + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) S[x] = 0.f;
        }
        if (snap0) store_state_row(p.pool, r.tslot, p.H, it.h, i, col0, S);
        if (r.nchunks > 0) {
            if (npro == 0) store_state_split(s_hi, s_lo, i, col0 >> 6, (col0 >> 5) & 1, S);
            uint32_t w[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) w[x] = __float_as_uint(S[x] * d0s);
            tmem_st32(t_s + (uint32_t)col0, w);
        } else if (!it.prefix()) {
            store_state_row(p.pool, r.slot, p.H, it.h, i, col0, S);
        }
    }
    if (r.nchunks > 0) tmem_st_wait();
    if (it.signals()) {
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            atomicAdd(&counters[r.b * p.H + it.h], 1);
        }
    }
}

// An item's end, from TMEM (left unscaled by its last chunk): the final state into the pool slot
// (last segment only; for a cut request with a prefix once every other segment has read S0), and
// the snapshot when it is at the segment's end.
template <bool kEx>
__device__ __forceinline__ void end_seg(const ExtendParams &p, const SegItem &it, uint32_t t_s,
                                        int col_base, int i, int lane, bool snap,
                                        const int *counters, uint64_t limit,
                                        volatile int *abort_flag) {
    const bool fin = it.last();
    if (!fin && !(kEx && snap)) return;
    if (fin && it.r.nseg > 1 && it.prefix()) {
        bool ok = true;
        if (lane == 0) {
            const int want = kEpiWarps * (it.r.nseg - 1);
            const int *cnt = counters + it.r.b * p.H + it.h;
            const uint64_t t0 = globaltimer_ns();
            while (true) {
                int v;
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
                if (v >= want) break;
                if (*abort_flag || globaltimer_ns() - t0 > limit) {
                    if (!*abort_flag) atomicOr(p.err, ERR_BIT_TIMEOUT);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
            }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return;
    }
#pragma unroll 1
    for (int sub = 0; sub < 2; ++sub) {
        const int col0 = col_base + sub * 32;
        uint32_t w[32];
        tmem_ld32(t_s + (uint32_t)col0, w);
        tmem_ld_wait_regs(w);
        float S[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) S[x] = __uint_as_float(w[x]);
        if (fin) store_state_row(p.pool, it.r.slot, p.H, it.h, i, col0, S);
        if (kEx && snap) store_state_row(p.pool, it.r.tslot, p.H, it.h, i, col0, S);
    }
}

// kEx: the options variant (state-tracking snapshots, caller-given output strides)
template <bool kEx>
__global__ void __launch_bounds__(kThreads, 1)
    extend_bal_kernel(const __grid_constant__ CUtensorMap tq,
                      const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const ExtendParams p,
                      const SegHeader *hdr, const SegRec *recs, int *counters) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw);
    Bars *bars = reinterpret_cast<Bars *>(sm + OFF_BAR);
    // Prologue chunks have a barrier pair per lambda-K lo buffer (stream index parity): kp_ready
    // (epilogue -> MMA: lambda K written) and pro_done (MMA -> epilogue: the chunk's MMAs done).
    // With two buffers the epilogue may run two prologue chunks ahead of the MMA thread, so one
    // barrier for both would complete twice before a wait and the parity would not tell; the
    // segments' chunks keep k_ready, counted over those chunks only.
    uint64_t *pro_done = reinterpret_cast<uint64_t *>(sm + OFF_BAR + sizeof(Bars));
    uint64_t *kp_ready = pro_done + 2;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;
    const int H = p.H;
    auto no_finish = [](const SegItem &) {};

    // Set-up touches only this CTA's shared and tensor memory, so it runs while the plan is
    // still being made; everything after the wait sees the plan (and the previous kernel's
    // writes).  The next kernel is let in at this CTA's end.

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        mbar_init(&bars->v_full, 1);
        mbar_init(&bars->v_empty, 1);
        mbar_init(&bars->a_full, 1);
        mbar_init(&bars->k_ready, kEpiWarps);
        mbar_init(&bars->p_ready, kEpiWarps);
        mbar_init(&bars->s_ready, kEpiWarps);
        mbar_init(&bars->o_free, kEpiWarps);
        mbar_init(&bars->u_full, 1);
        mbar_init(&bars->o_full, 1);
        mbar_init(&bars->drain, 1);
        mbar_init(&pro_done[0], 1);
        mbar_init(&pro_done[1], 1);
        mbar_init(&kp_ready[0], kEpiWarps);
        mbar_init(&kp_ready[1], kEpiWarps);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    const uint32_t tbase = bars->tmem_base;
    volatile int *abort_flag = &bars->abort_flag;
    const int nrec = hdr->nrec;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            Issued is{0, 0, 0};
            SegWalk walk;
            walk.start(recs, nrec, H);
            SegItem it;
            Uses u;
            bool ok = true;
            while (ok && walk.take(recs, nrec, H, it, no_finish)) {
                const int x = it.h * kHeadDim;
                const int y_req = it.r.y0 - it.r.a;  // the request's first token
                const int npro = it.npro();
                for (int pc = 0; pc < npro && ok; ++pc)
                    ok = produce_kv(bars, sm, tk, tv, u, y_req + pc * C, x, limit, abort_flag,
                                    p.err, is);
                int ys = 0;
                for (int c = 0; c < it.r.nchunks && ok; ++c) {
                    const int y = it.r.y0 + (kEx ? ys : c * C);
                    if (kEx) ys += chunk_len(true, ys, it.r.sp, it.r.len);
                    ok = produce_qkv(bars, sm, tq, tk, tv, u, y, x, limit, abort_flag, p.err, is);
                }
            }
            produce_drain(bars, is, p.err);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t s_base = smem_u32(sm);
            const uint32_t idA = idesc_bf16_f32(128, 128, false, false);
            const uint32_t idI = idesc_bf16_f32(128, kHeadDim, false, true);
            const uint32_t idU = idesc_bf16_f32(128, kHeadDim, true, true);
            const uint64_t dQ = sdesc_sw128(s_base + OFF_Q, 16, 1024);
            const uint64_t dK0 = sdesc_sw128(s_base + OFF_K, 16, 1024);
            const uint64_t dKt0 = sdesc_sw128(s_base + OFF_K, 16384, 1024);
            const uint64_t dKlo = sdesc_sw128(s_base + OFF_KLO, 16384, 1024);
            const uint64_t dV = sdesc_sw128(s_base + OFF_V, 16384, 1024);
            const uint64_t stage_step = SZ_T >> 4;
            const uint64_t dHi = sdesc_sw128(s_base + OFF_SHI, 16384, 1024);
            const uint64_t dLo = sdesc_sw128(s_base + OFF_SLO, 16384, 1024);
            // prologue chunks with an odd stream index: V in the Q buffer, lambda K lo in S_hi's
            const uint64_t dVq = sdesc_sw128(s_base + OFF_Q, 16384, 1024);
            SegWalk walk;
            walk.start(recs, nrec, H);
            SegItem it;
            Uses u;
            int gq = 0, ns = 0;
            bool ok = true;
            // S += (lambda K)_hi^T V + (lambda K)_lo^T V with K in stage st
            auto update = [&](int st, uint64_t dlo, uint64_t dv) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + TM_S, dKt0 + st * stage_step + mnofs(kk), dv + mnofs(kk),
                             idU, 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + TM_S, dlo + mnofs(kk), dv + mnofs(kk), idU, 1);
            };
            while (ok && walk.take(recs, nrec, H, it, no_finish)) {
                const int npro = it.npro();
                if (npro > 0) {
                    // the seed (e^{-s a} S0 in TMEM) is written, the last item's state read
                    if (!(ok = wait_bar(&bars->s_ready, ns & 1, limit, abort_flag, p.err))) break;
                    ++ns;
                    for (int pc = 0; pc < npro; ++pc) {
                        const int st = u.gk & 1;
                        const bool odd = (u.gp & 1) != 0;
                        if (!(ok = wait_bar(&kp_ready[u.gp & 1], (u.gp >> 1) & 1, limit,
                                            abort_flag, p.err)) ||
                            !(ok = odd ? wait_bar(&bars->q_full, u.nq & 1, limit, abort_flag, p.err)
                                       : wait_bar(&bars->v_full, u.nv & 1, limit, abort_flag,
                                                  p.err)))
                            break;
                        tc_fence_after();
                        update(st, odd ? dHi : dKlo, odd ? dVq : dV);
                        mma_commit(&bars->k_empty[st]);
                        mma_commit(odd ? &bars->q_empty : &bars->v_empty);
                        mma_commit(&pro_done[u.gp & 1]);
                        ++u.gk;
                        if (odd) ++u.nq; else ++u.nv;
                        ++u.gp;
                    }
                    if (!ok) break;
                }
                for (int c = 0; c < it.r.nchunks; ++c, ++u.gk, ++u.nq, ++u.nv, ++gq) {
                    const int st = u.gk & 1;
                    const int gk = u.gk;
                    // MMA1: A = Q K^T
                    if (!(ok = wait_bar(&bars->q_full, u.nq & 1, limit, abort_flag, p.err)) ||
                        !(ok = wait_bar(&bars->k_full[st], (gk >> 1) & 1, limit, abort_flag,
                                        p.err)))
                        break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tbase + TM_A, dQ + kofs(kk), dK0 + st * stage_step + kofs(kk),
                                 idA, kk > 0);
                    mma_commit(&bars->a_full);
                    // MMA2: Oint = Q S_hi + Q S_lo, after the state pass and the last output pass
                    if (!(ok = wait_bar(&bars->s_ready, ns & 1, limit, abort_flag, p.err)) ||
                        (gq >= 1 &&
                         !(ok = wait_bar(&bars->o_free, (gq - 1) & 1, limit, abort_flag, p.err))))
                        break;
                    ++ns;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tbase + TM_OI, dQ + kofs(kk), dHi + mnofs(kk), idI, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tbase + TM_OI, dQ + kofs(kk), dLo + mnofs(kk), idI, 1);
                    mma_commit(&bars->q_empty);
                    // MMA4: the state update, once lambda K and V are in
                    if (!(ok = wait_bar(&bars->k_ready, gq & 1, limit, abort_flag, p.err)) ||
                        !(ok = wait_bar(&bars->v_full, u.nv & 1, limit, abort_flag, p.err)))
                        break;
                    tc_fence_after();
                    update(st, dKlo, dV);
                    mma_commit(&bars->u_full);
                    mma_commit(&bars->k_empty[st]);
                    // MMA3: Ointra = P_hi V + P_lo V, P from TMEM
                    if (!(ok = wait_bar(&bars->p_ready, gq & 1, limit, abort_flag, p.err))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16_tmem_a(tbase + TM_OP, tbase + TM_A + p_col(kk), dV + mnofs(kk),
                                       idI, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16_tmem_a(tbase + TM_OP, tbase + TM_A + p_col(kk) + 16u,
                                       dV + mnofs(kk), idI, 1);
                    mma_commit(&bars->o_full);
                    mma_commit(&bars->v_empty);
                }
            }
            mma_commit(&bars->drain);
            int dummy = 0;
            wait_bar(&bars->drain, 0, kDrainLimitNs, &dummy, p.err);
        }
    } else {
        // ------------------------------------------------------------------ epilogue warps
        const int q = warp & 3;
        const int cw = warp >> 2;
        const int col_base = cw * 64;
        const int i = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const uint32_t t_s = tbase + lane_off + TM_S;
        const int pb0 = cw ? (q + 2) >> 1 : 0;
        const int pb1 = cw ? q + 1 : (q + 2) >> 1;
        const int zb0 = q + 1;
        const int zb1 = cw == 1 ? 4 : q + 1;
        const int ku0 = kKUnits * warp;
        uint8_t *s_hi = sm + OFF_SHI;
        uint8_t *s_lo = sm + OFF_SLO;
        const size_t row_stride = kEx ? (size_t)p.out_rs : (size_t)H * kHeadDim;
        const size_t head_stride = kEx ? (size_t)p.out_hs : (size_t)kHeadDim;
        auto finish = [&](const SegItem &z) {
            seed_seg<kEx>(p, z, t_s, col_base, s_hi, s_lo, i, lane, counters);
        };

        SegWalk walk;
        walk.start(recs, nrec, H);
        SegItem cur;
        bool have = walk.take(recs, nrec, H, cur, finish);
        if (have) seed_seg<kEx>(p, cur, t_s, col_base, s_hi, s_lo, i, lane, counters);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_ready);

        bool ok = true;
        int gk = 0, gq = 0, gp = 0;
        while (have && ok) {
            const float slope = p.slopes[cur.h];
            const bool run = slope <= kRunMaxSlope;
            const float grow = run ? expf(slope) : 1.f;
            const float gam = expf(-slope * (float)(i + 1)) * kScale;
            const float dn_full = expf(-slope * (float)C);
            LamSplitBf lam_full[kKUnits];
#pragma unroll
            for (int u = 0; u < kKUnits; ++u)
                lam_full[u] =
                    lam_split_bf16(expf(-slope * (float)(C - 1 - (((ku0 + u) >> 2) * 32 + lane))));
            const float f_p0 = pb0 < pb1 ? expf(-slope * (float)(i - 32 * pb0)) * kScale : 0.f;
            const float f_p1 =
                pb0 + 1 < pb1 ? expf(-slope * (float)(i - 32 * (pb0 + 1))) * kScale : 0.f;
            const SegItem it = cur;
            const int npro = it.npro();
            // ---- prologue: S_a = e^{-s a} S0 + sum over the first a tokens, then the first
            // chunk's operands from it
            if (npro > 0) {
                for (int pc = 0; pc < npro; ++pc, ++gk, ++gp) {
                    const int st = gk & 1;
                    // lambda K lo alternates between its buffer and S_hi's (idle until the
                    // prologue ends); a buffer is free again once the MMAs of the prologue chunk
                    // before last are done.  At an item's start both are: their last readers, the
                    // previous chunk's MMA4 and MMA2, were waited for in its state pass.
                    if (pc >= 2 && !(ok = warp_wait_bar(&pro_done[gp & 1], ((gp - 2) >> 1) & 1,
                                                        limit, abort_flag, p.err)))
                        break;
                    if (!(ok = warp_wait_bar(&bars->k_full[st], (gk >> 1) & 1, limit, abort_flag,
                                             p.err)))
                        break;
                    lamk_pro_pass(sm, st, (gp & 1) ? OFF_SHI : OFF_KLO, ku0, lane, slope,
                                  it.r.a - (pc + 1) * C);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&kp_ready[gp & 1]);
                }
                if (!ok) break;
                // the last prologue chunk's MMAs done (so every earlier one's): S_a is complete
                if (!(ok = warp_wait_bar(&pro_done[(gp - 1) & 1], ((gp - 1) >> 1) & 1, limit,
                                         abort_flag, p.err)))
                    break;
                tc_fence_after();
                const int r0 = chunk_len(kEx, 0, it.r.sp, it.r.len);
                const float d0 = r0 == C ? dn_full : expf(-slope * (float)r0);
                const bool snap = kEx && it.r.sp == 0;
                state_pass<kEx, 2>(t_s, col_base, s_hi, s_lo, i, d0, snap, p.pool, it.r.tslot, H,
                                   it.h, 0);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->s_ready);
            }
            bool have_nx = false;
            int cs_next = 0;
            for (int c = 0; c < it.r.nchunks; ++c, ++gk, ++gq) {
                const int st = gk & 1;
                const int cs = kEx ? cs_next : c * C;
                const int r = chunk_len(kEx, cs, it.r.sp, it.r.len);
                if (kEx) cs_next = cs + r;
                const bool last = c + 1 == it.r.nchunks;
                if (last && walk.more && walk.nxt.prefix()) {
                    const float *nrow = p.pool + (((size_t)walk.nxt.r.slot * H + walk.nxt.h) *
                                                      kHeadDim + i) * kHeadDim + (size_t)col_base;
                    prefetch_l2(nrow);
                    prefetch_l2(nrow + 32);
                }

                if (!(ok = warp_wait_bar(&bars->a_full, gq & 1, limit, abort_flag, p.err))) break;
                tc_fence_after();
                lamk_pass(sm, st, ku0, lane, r, slope, lam_full);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->k_ready);
                p_pass<false>(tbase + lane_off + TM_A, i, pb0, pb1, zb0, zb1, nullptr, slope, run,
                              grow, f_p0, f_p1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_ready);

                if (!(ok = warp_wait_bar(&bars->u_full, gq & 1, limit, abort_flag, p.err))) break;
                tc_fence_after();
                if (!last) {
                    const int r_next = chunk_len(kEx, cs + r, it.r.sp, it.r.len);
                    const float dn = r_next == C ? dn_full : expf(-slope * (float)r_next);
                    state_pass<kEx, 2>(t_s, col_base, s_hi, s_lo, i, dn, kEx && cs + r == it.r.sp,
                                       p.pool, it.r.tslot, H, it.h, 0);
                } else {
                    // MMA4 and (by issue order) MMA2 of the item's last chunk are done: its state
                    // leaves TMEM, and the next item's start takes the operand tiles and TMEM
                    end_seg<kEx>(p, it, t_s, col_base, i, lane, kEx && cs + r == it.r.sp,
                                 counters, limit, abort_flag);
                    SegItem nx;
                    have_nx = walk.take(recs, nrec, H, nx, finish);
                    if (have_nx) {
                        seed_seg<kEx>(p, nx, t_s, col_base, s_hi, s_lo, i, lane, counters);
                        cur = nx;
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->s_ready);

                if (!(ok = warp_wait_bar(&bars->o_full, gq & 1, limit, abort_flag, p.err))) break;
                tc_fence_after();
                out_pass<2>(tbase + lane_off, col_base, gam, lane, q, r, p.out, it.r.y0 + cs,
                            row_stride, (size_t)it.h * head_stride);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->o_free);
            }
            have = have_nx;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    if (warp == kMmaWarp) {
        __syncwarp();
        tmem_dealloc(tbase, kTmemCols);
    }
}

static_assert(sizeof(Bars) + 4 * sizeof(uint64_t) <= SZ_BAR, "barrier block with the prologue's");

}  // namespace

size_t bal_scratch_bytes(int B, int H) {
    return sizeof(SegHeader) + sizeof(SegRec) * (size_t)kMaxBalRecs +
           (((size_t)B * H * sizeof(int) + 15) & ~(size_t)15);
}

cudaError_t launch_extend_bal(const ExtendParams &p, void *scratch, int ctas, cudaStream_t stream) {
    if (ctas <= 0 || p.B <= 0) return cudaSuccess;
    if (scratch == nullptr || p.group != 1 || p.seg_len > 0 || p.B > kMaxBalRequests ||
        (reinterpret_cast<uintptr_t>(scratch) & 15) != 0)
        return cudaErrorInvalidValue;
    SegHeader *hdr = static_cast<SegHeader *>(scratch);
    SegRec *recs = reinterpret_cast<SegRec *>(static_cast<char *>(scratch) + sizeof(SegHeader));
    int *counters = reinterpret_cast<int *>(static_cast<char *>(scratch) + sizeof(SegHeader) +
                                            sizeof(SegRec) * (size_t)kMaxBalRecs);
    cudaError_t e = launch_pdl(seg_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, p, ctas,
                               hdr, recs, counters);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tk, tv;
    memset(&tq, 0, sizeof(tq));
    memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv));
    if (p.T > 0) {
        if (!make_token_map_full(&tq, p.q, p.T, p.H) || !make_token_map_full(&tk, p.k, p.T, p.H) ||
            !make_token_map_full(&tv, p.v, p.T, p.H))
            return cudaErrorInvalidValue;
    }
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static bool configured[64] = {false};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!configured[dev]) {
            e = cudaFuncSetAttribute(extend_bal_kernel<false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(extend_bal_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    if (p.track_lens != nullptr || p.out_rs != (long long)p.H * kHeadDim || p.out_hs != kHeadDim)
        return launch_pdl(extend_bal_kernel<true>, dim3((unsigned)ctas), dim3(kThreads),
                          kSmemBytes, stream, tq, tk, tv, p, (const SegHeader *)hdr,
                          (const SegRec *)recs, counters);
    return launch_pdl(extend_bal_kernel<false>, dim3((unsigned)ctas), dim3(kThreads), kSmemBytes,
                      stream, tq, tk, tv, p, (const SegHeader *)hdr, (const SegRec *)recs,
                      counters);
}

}  // namespace la
