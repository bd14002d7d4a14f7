// la_extend_w.cu -- chunked seg_la extend on the 5th-generation tensor cores, one CTA per
// (request, head): every MMA is 128 columns wide and the masked score matrix P lives in tensor
// memory.
//
// Method: page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section
// "独立参考实现：逐 token 递推公式": per head, S_t = S_{t-1} e^{-s} + outer(k_t, v_t) and
// o_t = (q_t @ S_t) D^-0.5, over each request's tokens, from the request's pool state (or zero),
// final state written back.  A request with a state-tracking snapshot (same page, section
// "额外覆盖") has its chunk grid restarted at the tracked token, so the snapshot is the state at a
// chunk boundary.
//
// Chunked form (exact up to rounding; local token indices i, j in [0, r), S the state before the
// chunk):
//   o_i    = D^-0.5 gamma_i (Q S)_i  +  ((Q K^T o Dm) D^-0.5 V)_i,
//            gamma_i = e^{-s (i+1)},  Dm_ij = e^{-s (i-j)} if j <= i, else 0
//   S_next = e^{-s r} S  +  K^T diag(lambda) V,       lambda_j = e^{-s (r-1-j)}
//
// Why one CTA per head.  An M = 128 tcgen05.mma costs about the same whether N is 64 or 128, so
// covering all 128 value columns in one CTA halves the MMA instructions per head and chunk, and
// the score matrix Q K^T and its mask are built once per head instead of once per column half.
// What it costs is storage: the value tile doubles, so Q and V have a single shared-memory buffer
// each (K keeps two), P moves into tensor memory in place of Q K^T, and the state update
// accumulates straight into the fp32 master state in tensor memory (pre-scaled by the next
// chunk's decay) instead of into a separate U buffer.
//
// Precision.  Every product runs in bf16 with fp32 accumulation, and the three operands that are
// computed in the kernel carry a bf16 pair hi + lo (about 2^-17): the state for Q S, P for P V,
// and lambda K for the state update.  A single 16-bit lambda K rounds each term of the state
// update, which a slowly decaying head sums over thousands of tokens; a single bf16 P or state
// operand breaks the parity bound outright.  V and K are used as loaded.
//
// Roles (320 threads):
//   warp 8      TMA producer: K of each chunk into a two-stage ring; Q and V into their buffers
//               once the previous chunk's products with them are done;
//   warp 9      TMEM allocator and MMA issuer (one thread), all bf16 with fp32 accumulation:
//                 MMA1  A       = Q K^T                            -> TMEM (128 columns)
//                 MMA2  Oint    = Q S_hi + Q S_lo                  -> TMEM (NV columns)
//                 MMA4  S      += (lambda K)_hi^T V + (lambda K)_lo^T V   -> TMEM (the state)
//                 MMA3  Ointra  = P_hi V + P_lo V  (P from TMEM)   -> TMEM (NV columns)
//   warps 0-7   first phase: two units of lambda K each (32 rows x 32 columns; hi in place, lo
//               into its own buffer), then the P blocks of their TMEM lane quarter (warp % 4):
//               P = A o Dm D^-0.5 for 32 keys as hi + lo over that block's 32 columns of A (every
//               read of a row happens in the warp that overwrites it); then, per half of the
//               CTA's NV value columns (warp / 4): the state pass (S to bf16 hi + lo in shared memory for MMA2, snapshot
//               if tracked, S times the next chunk's decay back to TMEM) and the output pass
//               (gamma D^-0.5 Oint + Ointra -> bf16 -> global), after which Oint and Ointra are
//               released to the next chunk's MMA2 and MMA3.  The per-row decay factors of full
//               chunks are read from the table once, before the first chunk.
// TMEM (512 columns): A / P 128, Oint 128, Ointra 128, S 128 (NV = 128 value columns; a CTA of
// the column split below uses the first 64 of Oint, Ointra and S).
//
// Column split.  When one CTA per (request, head) leaves SMs idle, the longest requests run as two
// CTAs per head, each on one 64-column half of the values (NV = 64): S[:, cols] and out[:, cols]
// depend only on V[:, cols], so the halves share nothing.  A half repeats the lambda-K units, P
// and MMA1 (they span all 128 key dimensions and keys) but runs MMA2, MMA4 and MMA3 with N = 64
// and halves the state and output passes, so its chunks are shorter and the longest request's
// chain no longer ends the kernel first.  The column count is a template parameter of the CTA's
// code path.
//
// Per chunk c, the MMA thread issues MMA2_c (after the state pass of c-1 and the output pass of
// c-1), MMA4_c (after K is scaled and V has landed), MMA3_c (after P), then MMA1_{c+1}.  The
// orders that make the buffer reuse safe: MMA1_{c+1} overwrites A/P after MMA3_c by issue order;
// P_c is written after MMA1_c is complete; the state pass of c rewrites S_hi/S_lo after u_full(c),
// which also covers MMA2_c; MMA4_c accumulates into S after the state pass of c-1 has scaled it;
// the lambda-K lo buffer is rewritten after MMA1_c, hence after MMA4_{c-1}; Q_{c+1} is loaded after
// MMA2_c (and so MMA1_c) is complete, V_{c+1} after MMA3_c.
//
// Every mbarrier wait is bounded (a globaltimer deadline).  A wait that runs out sets the error
// word and an abort flag; every role then leaves its loop, the producer waits for its own copies
// in flight and the MMA issuer for its MMAs, and the CTA frees its TMEM and exits.  No named
// barrier is used after the first wait of the kernel.
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "la_extend_tile.cuh"

namespace la {

namespace {

using namespace sm100;

// One CTA's work: request b, head h, segment g, value columns c0 .. c0 + NV - 1 (NV = 128, or 64
// under the column split).
template <bool kEx, int NV>
__device__ __forceinline__ void extend_cta(const CUtensorMap &tq, const CUtensorMap &tk,
                                           const CUtensorMap &tv, const ExtendParams &p,
                                           uint8_t *sm, const int g, const int h, const int b,
                                           const int c0_half) {
    constexpr int nv = NV;                               // value columns of this CTA
    const int c0 = NV == kHeadDim ? 0 : c0_half;         // its first value column
    Bars *bars = reinterpret_cast<Bars *>(sm + OFF_BAR);
    float *tab = reinterpret_cast<float *>(sm + OFF_TAB);
    float *tabp = reinterpret_cast<float *>(sm + OFF_TABP);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = p.H;
    // grouped-query heads: query head h reads kv head hk (k, v, slope, state); hk = h otherwise
    const int Hkv = p.Hkv;
    const int hk = p.group == 1 ? h : h / p.group;
    // with a group, every query head's CTA carries the kv head's state and the group's first one
    // writes it back
    const bool writes_state = p.group == 1 || hk * p.group == h;

    // Request geometry, checked before anything is allocated (the exit is CTA-uniform).
    const int slot = p.state_idx[b];
    const int t_req0 = p.cu_seqlens[b];
    const int t_req1 = p.cu_seqlens[b + 1];
    if (slot < 0 || slot >= p.num_slots) {
        if (threadIdx.x == 0 && g == 0) atomicOr(p.err, ERR_BIT_SLOT_RANGE);
        return;
    }
    if (t_req0 < 0 || t_req1 < t_req0 || t_req1 > p.T) {
        if (threadIdx.x == 0 && g == 0) atomicOr(p.err, ERR_BIT_SEQLENS);
        return;
    }
    // Segment [t0, t1) of the request: the whole request unless long requests are split.
    const int n_req = t_req1 - t_req0;
    // max_seqlen is the caller's bound on every request's length, and the split schedule has no
    // CTA for the segments past it: a longer request is reported and skipped, never half-written.
    if (n_req > p.max_seqlen) {
        if (threadIdx.x == 0 && g == 0) atomicOr(p.err, ERR_BIT_SEQLENS);
        return;
    }
    int nseg_b = 1, t0 = t_req0, t1 = t_req1;
    if (p.seg_len > 0) {
        nseg_b = n_req > 0 ? (n_req + p.seg_len - 1) / p.seg_len : 1;
        if (g >= nseg_b) return;
        t0 = t_req0 + g * p.seg_len;
        t1 = min(t_req1, t0 + p.seg_len);
    }
    const bool split = nseg_b > 1;
    const bool last_seg = g == nseg_b - 1;
    const int n = t1 - t0;
    // State tracking: the CTA whose segment holds token offset tl (the last segment when tl is
    // the request's end) restarts its chunk grid at that token (local offset sp) and stores the
    // state it carries at that boundary; every other CTA keeps the regular grid (sp = n + 1).
    int sp = n + 1;
    if (kEx && p.track_lens != nullptr) {
        const int tl = p.track_lens[b];
        const int tslot = p.track_idx[b];
        if (tl >= 0) {
            if (tl > n_req || tslot < 0 || tslot >= p.num_slots || tslot == slot) {
                if (threadIdx.x == 0 && g == 0) atomicOr(p.err, ERR_BIT_TRACK);
            } else {
                const int tloc = tl - (t0 - t_req0);
                if ((tloc >= 0 && tloc < n) || (tloc == n && last_seg)) sp = tloc;
            }
        }
    }
    const int nchunks = kEx && sp <= n ? (sp + C - 1) / C + (n - sp + C - 1) / C
                                       : (n + C - 1) / C;
    const uint64_t limit = p.wait_limit_ns;

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
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0 && nchunks > 0) {
        tma_prefetch_desc(&tq);
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
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            Issued is{0, 0, 0};
            int ys = 0;
            const int xq = h * kHeadDim;    // query head h in q
            const int xkv = hk * kHeadDim;  // its kv head in k and v
            for (int c = 0; c < nchunks; ++c) {
                const int y = t0 + (kEx ? ys : c * C);
                if (kEx) ys += chunk_len(true, ys, sp, n);
                if (!produce_chunk<nv>(bars, sm, tq, tk, tv, c, y, xq, xkv, c0, limit, abort_flag,
                                       p.err, is))
                    break;
            }
            produce_drain(bars, is, p.err);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            mma_loop<nv>(bars, tbase, s_base, nchunks, limit, abort_flag, p.err);
        }
    } else {
        // ------------------------------------------------------------------ epilogue warps
        const int q = warp & 3;            // TMEM lane quarter
        const int cw = warp >> 2;          // column slot for the state and output passes
        constexpr int nsubs = nv / (32 * kColWarps);  // 32-column parts per warp: 2, or 1 at nv = 64
        const int col_base = cw * 32 * nsubs;  // columns col_base .. col_base + 32 nsubs - 1 of
                                               // the CTA's nv (value column c0 + col)
        const int i = q * 32 + lane;       // row: token of the chunk (A, O) or k-dim (S)
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        // Work split of the chunk's first phase.  Every warp first scales kKUnits of the 16
        // lambda-K units (4 row groups x 4 column quarters), so that MMA4 can start early; then
        // lane quarter q's P blocks 0 .. q, split over its two warps (warp q the lower blocks,
        // warp q + 4 the upper ones), and the zero blocks above the diagonal (warp q + 4).
        const int pb0 = cw ? (q + 2) >> 1 : 0;
        const int pb1 = cw ? q + 1 : (q + 2) >> 1;
        const int zb0 = q + 1;
        const int zb1 = cw == 1 ? 4 : q + 1;
        const int ku0 = kKUnits * warp;  // units ku0 .. ku0 + kKUnits - 1

        const float slope = p.slopes[hk];
        for (int m = threadIdx.x; m <= C; m += kEpiThreads) {
            const float e = expf(-slope * (float)m);
            tab[m] = e;
            tabp[m] = e * kScale;
        }
        const bool run = slope <= kRunMaxSlope;       // false for NaN slopes too
        const float grow = run ? expf(slope) : 1.f;  // e^{s}: one step along a row of P
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");  // tables
        uint8_t *s_hi = sm + OFF_SHI;
        uint8_t *s_lo = sm + OFF_SLO;
        // this row's share of the pool state: value columns c0 + col_base .. + 32 nsubs - 1
        float *gstate = p.pool + (((size_t)slot * Hkv + hk) * kHeadDim + i) * kHeadDim +
                        (size_t)(c0 + col_base);
        {
            const int r0 = nchunks > 0 ? chunk_len(kEx, 0, sp, n) : 0;
            const float d0s = expf(-slope * (float)r0);
#pragma unroll 1
            for (int sub = 0; sub < nsubs; ++sub) {
                const int col0 = col_base + sub * 32;
                float S[32];
                if (split || p.group > 1) {
                    // From the workspace: S0 (its copy) for the first segment and for an unsplit
                    // request of a grouped call; for segment g >= 1 the start state
                    // e^{-s g seg} S0 + sum_{k < g P} e^{-s (g seg - (k+1) blk)} B_k, which the
                    // state scan left in block state g P - 1.
                    const size_t m = g == 0 ? 0 : (size_t)g * (p.seg_len / p.blk_len);
                    const float *w0 = p.ws + (((size_t)b * Hkv + hk) * (size_t)(1 + p.nblk) + m) *
                                                 (kHeadDim * kHeadDim) +
                                      (size_t)i * kHeadDim + c0 + col0;
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const float4 f = reinterpret_cast<const float4 *>(w0)[x];
                        S[4 * x] = f.x;
                        S[4 * x + 1] = f.y;
                        S[4 * x + 2] = f.z;
                        S[4 * x + 3] = f.w;
                    }
                } else if (p.prefix_mask[b]) {
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const float4 f =
                            *reinterpret_cast<const float4 *>(gstate + sub * 32 + 4 * x);
                        S[4 * x] = f.x;
                        S[4 * x + 1] = f.y;
                        S[4 * x + 2] = f.z;
                        S[4 * x + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) S[x] = 0.f;
                }
                if (kEx && sp == 0)
                    store_state_row(p.pool, p.track_idx[b], H, h, i, c0 + col0, S);
                store_state_split(s_hi, s_lo, i, col0 >> 6, (col0 >> 5) & 1, S);
                // TMEM holds e^{-s r_0} S_0, onto which MMA4 of chunk 0 accumulates
                uint32_t w[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) w[x] = __float_as_uint(S[x] * d0s);
                tmem_st32(tbase + lane_off + TM_S + (uint32_t)col0, w);
            }
            tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_ready);

        // output layout: packed [T][H*128] unless the options variant was given other strides
        const size_t row_stride = kEx ? (size_t)p.out_rs : (size_t)H * kHeadDim;
        const size_t head_stride = kEx ? (size_t)p.out_hs : (size_t)kHeadDim;
        bool ok = true;
        int cs_next = 0;
        // Factors that stay fixed for every full chunk, formed once in registers (a ragged chunk
        // forms its own): reading them from the table measured slower.
        const float gam = expf(-slope * (float)(i + 1)) * kScale;  // gamma_i D^-0.5
        const float dn_full = expf(-slope * (float)C);            // decay over a full chunk
        LamSplitBf lam_full[kKUnits];      // lambda of this warp's K units' rows, full chunk
#pragma unroll
        for (int k = 0; k < kKUnits; ++k)
            lam_full[k] =
                lam_split_bf16(expf(-slope * (float)(C - 1 - (((ku0 + k) >> 2) * 32 + lane))));
        // P start factors e^{-s (i - 32 cb)} D^-0.5 of this warp's (at most two) blocks
        const float f_p0 = pb0 < pb1 ? expf(-slope * (float)(i - 32 * pb0)) * kScale : 0.f;
        const float f_p1 =
            pb0 + 1 < pb1 ? expf(-slope * (float)(i - 32 * (pb0 + 1))) * kScale : 0.f;
        for (int c = 0; c < nchunks; ++c) {
            const int st = c & 1;
            // first token of the chunk and its length
            const int cs = kEx ? cs_next : c * C;
            const int r = chunk_len(kEx, cs, sp, n);
            if (kEx) cs_next = cs + r;

            if (!(ok = warp_wait_bar(&bars->a_full, c & 1, limit, abort_flag, p.err))) break;
            tc_fence_after();
            // ---- lambda K as a bf16 pair hi (in place) + lo: this warp's units of (32-row group,
            // 32-column quarter)
            lamk_pass(sm, st, ku0, lane, r, slope, lam_full);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->k_ready);
            // ---- P = A o Dm D^-0.5 into TMEM as bf16 pairs; blocks above the diagonal zeroed
            p_pass<true>(tbase + lane_off + TM_A, i, pb0, pb1, zb0, zb1, tabp, slope, run, grow,
                         f_p0, f_p1);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_ready);

            // ---- state: S_c is in TMEM once MMA4 is done; hi/lo copy for MMA2_{c+1}, then
            // e^{-s r_{c+1}} S_c back for MMA4_{c+1}
            if (!(ok = warp_wait_bar(&bars->u_full, c & 1, limit, abort_flag, p.err))) break;
            tc_fence_after();
            {
                const int r_next = c + 1 < nchunks ? chunk_len(kEx, cs + r, sp, n) : 0;
                const float dn = c + 1 >= nchunks ? 1.f
                                 : r_next == C   ? dn_full
                                                 : expf(-slope * (float)r_next);
                const bool snap = kEx && cs + r == sp;
                state_pass<kEx, nsubs>(tbase + lane_off + TM_S, col_base, s_hi, s_lo, i, dn, snap,
                                       p.pool, snap ? p.track_idx[b] : 0, H, h, c0);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_ready);

            // ---- out: o = gamma D^-0.5 Oint + Ointra -> bf16, 32 columns at a time
            if (!(ok = warp_wait_bar(&bars->o_full, c & 1, limit, abort_flag, p.err))) break;
            tc_fence_after();
            out_pass<nsubs>(tbase + lane_off, col_base, gam, lane, q, r, p.out, t0 + cs, row_stride,
                            (size_t)h * head_stride + c0);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->o_free);
        }
        // Final state write-back (also for zero-length requests).  Skipped after an abort: the
        // error word already reports the failure.  The last state pass left S unscaled.
        if (ok && !*abort_flag && last_seg && writes_state) {
#pragma unroll 1
            for (int sub = 0; sub < nsubs; ++sub) {
                uint32_t w[32];
                tmem_ld32(tbase + lane_off + TM_S + (uint32_t)(col_base + sub * 32), w);
                tmem_ld_wait_regs(w);
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    *reinterpret_cast<float4 *>(gstate + sub * 32 + 4 * x) = make_float4(
                        __uint_as_float(w[4 * x]), __uint_as_float(w[4 * x + 1]),
                        __uint_as_float(w[4 * x + 2]), __uint_as_float(w[4 * x + 3]));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Let the next kernel on the stream be scheduled only now: triggered at the start, its CTAs
    // sat on the SMs this grid's short requests freed while the long ones ran, and measured
    // slower (varlen batch 91-95 us against 88 us triggered here).
    pdl_trigger();
    if (warp == kMmaWarp) {
        __syncwarp();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// kEx: the options variant (state-tracking snapshots, caller-given output strides)
template <bool kEx>
__global__ void __launch_bounds__(kThreads, 1)
    extend_wide_kernel(const __grid_constant__ CUtensorMap tq,
                       const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const ExtendParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw);
    pdl_wait();  // the next kernel is let in from the end of extend_cta (or this CTA's exit)

    const int H = p.H;
    const int g = blockIdx.x % p.nseg;  // segment of the request (0 when not split)
    const int bh = blockIdx.x / p.nseg;
    int h = bh % H;
    int want = bh / H;  // the request's rank in decreasing length order when p.lpt is set
    // Column split: the p.csplit longest requests run as two CTAs per head, each on one 64-column
    // half of the values (CTAs 2 (rank H + h) + half), the other requests as one CTA per head.
    // The halves share nothing: S[:, cols] depends only on V[:, cols].
    int half = -1;
    if (p.csplit > 0) {
        const int x = blockIdx.x;  // no sequence split alongside
        if (x < 2 * p.csplit * H) {
            want = x / (2 * H);
            h = (x >> 1) % H;
            half = x & 1;
        } else {
            const int y = x - p.csplit * H;
            want = y / H;
            h = y % H;
        }
    }
    int b = want;
    if (p.lpt && p.order != nullptr) {
        b = p.order[want];  // ranked by the pre-pass
    } else if (p.lpt) {
        // Longest request first: CTAs are issued in index order, so taking requests in
        // decreasing length order (ties by index) keeps long requests from finishing last.
        __shared__ int s_req;
        for (int t = threadIdx.x; t < p.B; t += kThreads) {
            const int lt = p.cu_seqlens[t + 1] - p.cu_seqlens[t];
            int rank = 0;
            for (int u = 0; u < p.B; ++u) {
                const int lu = p.cu_seqlens[u + 1] - p.cu_seqlens[u];
                rank += (lu > lt) || (lu == lt && u < t);
            }
            if (rank == want) s_req = t;
        }
        __syncthreads();
        b = s_req;
    }


    // The value-column count is a compile-time constant of each CTA's code path.
    if (half < 0)
        extend_cta<kEx, kHeadDim>(tq, tk, tv, p, sm, g, h, b, 0);
    else
        extend_cta<kEx, kHeadDim / 2>(tq, tk, tv, p, sm, g, h, b, half * (kHeadDim / 2));
}

// ----------------------------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

}  // namespace

// [T][H*128] bf16, box of 64 columns x C rows, 128-byte swizzle; rows past T read as zero.
bool make_token_map_full(CUtensorMap *m, const void *ptr, int T, int H) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H * kHeadDim, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * kHeadDim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)C};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

cudaError_t launch_extend_wide(const ExtendParams &p, cudaStream_t stream) {
    const long long units =
        (long long)p.B * p.H * (p.seg_len > 0 ? p.nseg : 1) + (long long)p.csplit * p.H;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap tq, tk, tv;
    memset(&tq, 0, sizeof(tq));
    memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv));
    if (p.T > 0) {
        if (!make_token_map_full(&tq, p.q, p.T, p.H) ||
            !make_token_map_full(&tk, p.k, p.T, p.Hkv) ||
            !make_token_map_full(&tv, p.v, p.T, p.Hkv))
            return cudaErrorInvalidValue;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static bool configured[64] = {false};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!configured[dev]) {
            e = cudaFuncSetAttribute(extend_wide_kernel<false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(extend_wide_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    const ExtendParams pw = p;
    if (p.track_lens != nullptr || p.out_rs != (long long)p.H * kHeadDim || p.out_hs != kHeadDim)
        return launch_pdl(extend_wide_kernel<true>, dim3((unsigned)units), dim3(kThreads),
                          kSmemBytes, stream, tq, tk, tv, pw);
    return launch_pdl(extend_wide_kernel<false>, dim3((unsigned)units), dim3(kThreads),
                      kSmemBytes, stream, tq, tk, tv, pw);
}

}  // namespace la
