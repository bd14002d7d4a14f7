// la_extend_many.cu -- chunked seg_la extend for batches of more than one wave: a persistent grid
// of one CTA per SM, each working through its share of the (request, head) items as one stream
// of chunks.
//
// Method: page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section
// "独立参考实现：逐 token 递推公式" (per head, S_t = S_{t-1} e^{-s} + outer(k_t, v_t) and
// o_t = (q_t @ S_t) D^-0.5 from the request's pool state or zero, final state written back), in
// the chunked form that la_extend_w.cu states; state-tracking snapshots as in section "额外覆盖".
//
// Why a second kernel.  With more (request, head) pairs than SMs, one CTA per pair pays, per
// pair, the CTA's setup (barriers, tensor memory), the first loads of its state and tiles with
// the SM's pipes idle, and the write of its final state; for batches of short requests that
// costs about as much as their chunks.  A persistent CTA keeps its barriers and tensor memory and
// runs the chunks of all its items back to back: the TMA producer loads the next item's tiles
// while the epilogue finishes the current one, the MMA issuer sees one uninterrupted stream of
// chunks, and the next item's initial state is prefetched into L2 one chunk ahead.
//
// Items.  A pre-pass ranks the requests by decreasing length (ties by index) and writes each
// one's geometry record (first token, length, slot, prefix flag, tracked token, chunk count; a
// faulty request is reported there and marked invalid) at its rank.  Item rank r is head r % H of
// the request with rank r / H; the items are dealt to the G CTAs in snake order (CTA j takes
// ranks j, 2G - 1 - j, 2G + j, 4G - 1 - j, ...), which evens out the CTAs' totals.  Every role
// reads an item's record with one load, issued an item ahead.  Each item is computed exactly as
// the one-CTA-per-item kernel computes it, so the results do not depend on which kernel ran.
//
// Per chunk the roles, buffers, barriers and orders are those of la_extend_w.cu, with chunks
// counted over the CTA's whole stream (the barrier parities).  Between items, the state pass of
// an item's last chunk writes the item's final state (and a tracking snapshot at the request's
// end) instead of the next chunk's operands, and seeds the next item: S0 (its pool slot, or zero)
// as the bf16 pair for its first MMA2 and e^{-s r0} S0 in TMEM for its first MMA4.  Zero-length
// requests have no chunks; their final state (zero without a prefix; a prefix state stays as it
// is) and snapshot are written when the stream passes them.  Not here: the column split, the
// sequence split and grouped heads, which only the one-CTA-per-item kernel runs.
#include <string.h>

#include <mutex>

#include "la_extend_tile.cuh"

namespace la {

namespace {

// One (request, head) item of a CTA's stream: its request's record and the head.
struct Item {
    ItemRec r;
    int h;
    __device__ bool valid() const { return (r.flags & kRecValid) != 0; }
    __device__ bool prefix() const { return (r.flags & kRecPrefix) != 0; }
};

// Item k of this CTA (the load is issued here and used later); false when it has fewer than
// k + 1.
__device__ __forceinline__ bool load_item(const ExtendParams &p, int k, Item &it) {
    const long long G = gridDim.x, j = blockIdx.x;
    const long long rk = (k & 1) ? (long long)(k + 1) * G - 1 - j : (long long)k * G + j;
    if (rk >= (long long)p.B * p.H) return false;
    const int4 *src = reinterpret_cast<const int4 *>(p.recs + rk / p.H);
    const int4 x = __ldg(src), y = __ldg(src + 1);
    it.r = ItemRec{x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
    it.h = (int)(rk % p.H);
    return true;
}

// A role's walk over its CTA's items: take() moves to the next item that has chunks, handing the
// zero-length ones it passes to `finish`; the record of the item after it is loaded meanwhile.
struct ItemWalk {
    int k = 0;
    bool more = false;
    Item nxt;
    __device__ __forceinline__ void start(const ExtendParams &p) { more = load_item(p, 0, nxt); }
    template <class Finish>
    __device__ __forceinline__ bool take(const ExtendParams &p, Item &out, Finish finish) {
        while (more) {
            out = nxt;
            more = load_item(p, ++k, nxt);
            if (!out.valid()) continue;
            if (out.r.nchunks > 0) return true;
            finish(out);
        }
        return false;
    }
};

// This thread's rows of an item's initial state S0 (pool slot with a prefix, else zero), columns
// col_base .. col_base + 63: a tracking snapshot at token 0; then, for an item with chunks, the
// bf16 pair for its first MMA2 and e^{-s r0} S0 into TMEM for its first MMA4, or, for a
// zero-length item without a prefix, its (zero) final state.
template <bool kEx>
__device__ __forceinline__ void seed_state(const ExtendParams &p, const Item &it, uint32_t t_s,
                                           int col_base, uint8_t *s_hi, uint8_t *s_lo, int i) {
    const ItemRec &r = it.r;
    const bool snap0 = kEx && r.sp == 0;
    if (r.nchunks == 0 && !snap0 && it.prefix()) return;  // the slot already holds the state
    const float slope = p.slopes[it.h];
    const int r0 = r.nchunks > 0 ? chunk_len(kEx, 0, r.sp, r.n) : 0;
    const float d0s = expf(-slope * (float)r0);
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
            store_state_split(s_hi, s_lo, i, col0 >> 6, (col0 >> 5) & 1, S);
            uint32_t w[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) w[x] = __float_as_uint(S[x] * d0s);
            tmem_st32(t_s + (uint32_t)col0, w);
        } else if (!it.prefix()) {
            store_state_row(p.pool, r.slot, p.H, it.h, i, col0, S);
        }
    }
    if (r.nchunks > 0) tmem_st_wait();
}

// Where box bx (state columns 32 bx .. 32 bx + 31, fp32, 128-byte swizzled) of an S0 loaded
// through the staging tiles lands: each box over the rows that will hold the same columns' bf16
// hi or lo, so that a thread converting its row overwrites only values it has read itself.
__device__ __forceinline__ uint32_t s0_box_offset(int bx) {
    return (uint32_t)((bx & 1) * 32768 + (bx >> 1) * 16384);
}

// The start of item it (with chunks and a prefix) from its S0 in the staging tiles: this thread's
// row i, columns col_base .. col_base + 63 (boxes 2 cw and 2 cw + 1), read whole before it is
// overwritten by its bf16 pair for the first MMA2; e^{-s r0} S0 into TMEM for the first MMA4.
__device__ __forceinline__ void seed_from_tiles(const ExtendParams &p, const Item &it,
                                                uint32_t t_s, int col_base, uint8_t *s_hi,
                                                uint8_t *s_lo, int i) {
    float S[64];
#pragma unroll
    for (int sub = 0; sub < 2; ++sub) {
        const uint8_t *row = s_hi + s0_box_offset((col_base >> 5) + sub) + i * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 f = *reinterpret_cast<const float4 *>(row + ((c ^ (i & 7)) << 4));
            S[sub * 32 + 4 * c] = f.x;
            S[sub * 32 + 4 * c + 1] = f.y;
            S[sub * 32 + 4 * c + 2] = f.z;
            S[sub * 32 + 4 * c + 3] = f.w;
        }
    }
    const float d0s = expf(-p.slopes[it.h] * (float)chunk_len(false, 0, it.r.sp, it.r.n));
#pragma unroll
    for (int sub = 0; sub < 2; ++sub) {
        const int col0 = col_base + sub * 32;
        store_state_split(s_hi, s_lo, i, col0 >> 6, (col0 >> 5) & 1, S + sub * 32);
        uint32_t w[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) w[x] = __float_as_uint(S[sub * 32 + x] * d0s);
        tmem_st32(t_s + (uint32_t)col0, w);
    }
    tmem_st_wait();
}

// This thread's row of an item's final state from TMEM (left unscaled by its last chunk) into the
// staging tiles for the TMA store: four boxes of [128 rows][32 fp32 columns], 16 KiB apart, each
// row's eight 16-byte chunks placed with the 128-byte swizzle the state map uses.
__device__ __forceinline__ void stage_final_state(uint32_t t_s, int col_base, int i, uint8_t *stg) {
#pragma unroll 1
    for (int sub = 0; sub < 2; ++sub) {
        const int col0 = col_base + sub * 32;
        uint32_t w[32];
        tmem_ld32(t_s + (uint32_t)col0, w);
        tmem_ld_wait_regs(w);
        uint8_t *row = stg + (col0 >> 5) * 16384 + i * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4 *>(row + ((c ^ (i & 7)) << 4)) =
                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}

// kEx: the options variant (state-tracking snapshots, caller-given output strides)
template <bool kEx>
__global__ void __launch_bounds__(kThreads, 1)
    extend_many_kernel(const __grid_constant__ CUtensorMap tq,
                       const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv,
                       const __grid_constant__ CUtensorMap tsm, const ExtendParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw);
    pdl_wait();  // the next kernel is let in at this CTA's end
    Bars *bars = reinterpret_cast<Bars *>(sm + OFF_BAR);
    // The hand-over of a finished item's state: stg_ready (the epilogue warps have staged their
    // rows of it in the S_hi / S_lo tiles) and stg_free (the TMA stores have read the tiles, which
    // the next item's start may overwrite).
    uint64_t *stg_ready = reinterpret_cast<uint64_t *>(sm + OFF_BAR + sizeof(Bars));
    uint64_t *stg_free = stg_ready + 1;
    // s0_full: the next item's S0 has landed in the staging tiles (a TMA load, plain variant)
    uint64_t *s0_full = stg_ready + 2;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;
    auto no_finish = [](const Item &) {};

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
        mbar_init(stg_ready, kEpiWarps);
        mbar_init(stg_free, 1);
        mbar_init(s0_full, 1);
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
        tma_prefetch_desc(&tsm);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bars->tmem_base;
    volatile int *abort_flag = &bars->abort_flag;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            Issued is{0, 0, 0};
            ItemWalk walk;
            walk.start(p);
            Item it;
            int gc = 0;
            bool ok = true;
            while (ok && walk.take(p, it, no_finish)) {
                const int x = it.h * kHeadDim;
                int ys = 0;
                for (int c = 0; c < it.r.nchunks; ++c, ++gc) {
                    const int y = it.r.t0 + (kEx ? ys : c * C);
                    if (kEx) ys += chunk_len(true, ys, it.r.sp, it.r.n);
                    if (!(ok = produce_chunk<kHeadDim>(bars, sm, tq, tk, tv, gc, y, x, x, 0, limit,
                                                       abort_flag, p.err, is)))
                        break;
                }
            }
            produce_drain(bars, is, p.err);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA issuer
        // the CTA's chunk count, its items' records read by the warp's lanes in parallel
        int total = 0;
        for (int k = lane;; k += 32) {
            Item it;
            if (!load_item(p, k, it)) break;
            if (it.valid()) total += it.r.nchunks;
        }
        total = __reduce_add_sync(0xffffffffu, total);
        if (lane == 0) mma_loop<kHeadDim>(bars, tbase, smem_u32(sm), total, limit, abort_flag, p.err);
    } else {
        // ------------------------------------------------------------------ epilogue warps
        const int q = warp & 3;     // TMEM lane quarter
        const int cw = warp >> 2;   // column slot for the state and output passes
        const int col_base = cw * 64;
        const int i = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const uint32_t t_s = tbase + lane_off + TM_S;
        // the chunk's first phase split as in the one-CTA-per-item kernel
        const int pb0 = cw ? (q + 2) >> 1 : 0;
        const int pb1 = cw ? q + 1 : (q + 2) >> 1;
        const int zb0 = q + 1;
        const int zb1 = cw == 1 ? 4 : q + 1;
        const int ku0 = kKUnits * warp;
        uint8_t *s_hi = sm + OFF_SHI;
        uint8_t *s_lo = sm + OFF_SLO;
        const size_t row_stride = kEx ? (size_t)p.out_rs : (size_t)p.H * kHeadDim;
        const size_t head_stride = kEx ? (size_t)p.out_hs : (size_t)kHeadDim;
        auto finish = [&](const Item &z) { seed_state<kEx>(p, z, t_s, col_base, s_hi, s_lo, i); };

        ItemWalk walk;
        walk.start(p);
        Item cur;
        bool have = walk.take(p, cur, finish);
        if (have) seed_state<kEx>(p, cur, t_s, col_base, s_hi, s_lo, i);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_ready);

        bool ok = true;
        int gc = 0;
        int nhand = 0;  // hand-overs so far (the staging barriers' phases)
        int nload = 0;  // S0 loads through the staging tiles so far (s0_full's phases)
        int s0_issued = 0;  // of them issued (thread 0): an abort may leave one unwaited
        while (have && ok) {
            // the item's factors, as in the one-CTA-per-item kernel
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
            const ItemRec r_cur = cur.r;
            const int h_cur = cur.h;
            bool have_nx = false;
            int cs_next = 0;
            for (int c = 0; c < r_cur.nchunks; ++c, ++gc) {
                const int st = gc & 1;
                const int cs = kEx ? cs_next : c * C;
                const int r = chunk_len(kEx, cs, r_cur.sp, r_cur.n);
                if (kEx) cs_next = cs + r;
                const bool last = c + 1 == r_cur.nchunks;
                // the next item's initial state rows into L2 a chunk ahead (its record is in)
                // the next item's initial state rows into L2 a chunk ahead (its record is in)
                if (last && walk.more && walk.nxt.valid() && walk.nxt.prefix()) {
                    const float *nrow = p.pool + (((size_t)walk.nxt.r.slot * p.H + walk.nxt.h) *
                                                      kHeadDim + i) * kHeadDim + (size_t)col_base;
                    prefetch_l2(nrow);
                    prefetch_l2(nrow + 32);
                }

                if (!(ok = warp_wait_bar(&bars->a_full, gc & 1, limit, abort_flag, p.err))) break;
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

                if (!(ok = warp_wait_bar(&bars->u_full, gc & 1, limit, abort_flag, p.err))) break;
                tc_fence_after();
                if (!last) {
                    const int r_next = chunk_len(kEx, cs + r, r_cur.sp, r_cur.n);
                    const float dn = r_next == C ? dn_full : expf(-slope * (float)r_next);
                    state_pass<kEx, 2>(t_s, col_base, s_hi, s_lo, i, dn, kEx && cs + r == r_cur.sp,
                                       p.pool, r_cur.tslot, p.H, h_cur, 0);
                } else {
                    // MMA4 and (by issue order) MMA2 of the item's last chunk are done: its final
                    // state leaves TMEM through the S_hi / S_lo tiles (free now) and TMA stores.
                    // While the stores read the tiles the epilogue runs the chunk's output pass
                    // (which does not touch them); then the next item's S0 takes the operand tiles
                    // and TMEM.  This keeps 64 KiB of global stores off the chain between the two
                    // items.
                    stage_final_state(t_s, col_base, i, s_hi);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(stg_ready);
                    if (threadIdx.x == 0 && wait_bar(stg_ready, nhand & 1, limit, abort_flag, p.err)) {
                        const int y = (cur.r.slot * p.H + cur.h) * kHeadDim;
#pragma unroll
                        for (int bx = 0; bx < 4; ++bx)
                            tma_store_2d(&tsm, s_hi + bx * 16384, bx * 32, y);
                        if (kEx && cs + r == r_cur.sp) {  // the snapshot at the request's end
                            const int ys = (cur.r.tslot * p.H + cur.h) * kHeadDim;
#pragma unroll
                            for (int bx = 0; bx < 4; ++bx)
                                tma_store_2d(&tsm, s_hi + bx * 16384, bx * 32, ys);
                        }
                        bulk_commit_group();
                    }
                    if (!(ok = warp_wait_bar(&bars->o_full, gc & 1, limit, abort_flag, p.err))) {
                        if (threadIdx.x == 0) mbar_arrive(stg_free);
                        break;
                    }
                    tc_fence_after();
                    out_pass<2>(tbase + lane_off, col_base, gam, lane, q, r, p.out, r_cur.t0 + cs,
                                row_stride, (size_t)h_cur * head_stride);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->o_free);
                    Item nx;
                    have_nx = walk.take(p, nx, finish);
                    // a prefix S0 comes in by one TMA load into the tiles, once the stores have
                    // read them (plain variant; the options variant loads it per thread)
                    const bool tma_s0 = !kEx && have_nx && nx.prefix();
                    if (threadIdx.x == 0) {
                        bulk_wait_group_read0();
                        if (tma_s0) {
                            const int y = (nx.r.slot * p.H + nx.h) * kHeadDim;
                            mbar_arrive_expect_tx(s0_full, 4 * 16384);
#pragma unroll
                            for (int bx = 0; bx < 4; ++bx)
                                tma_load_2d(s_hi + s0_box_offset(bx), &tsm, s0_full, bx * 32, y);
                            ++s0_issued;
                        }
                        mbar_arrive(stg_free);
                    }
                    if (!(ok = warp_wait_bar(stg_free, nhand & 1, limit, abort_flag, p.err))) break;
                    ++nhand;
                    if (tma_s0) {
                        if (!(ok = warp_wait_bar(s0_full, nload & 1, limit, abort_flag, p.err)))
                            break;
                        ++nload;
                        seed_from_tiles(p, nx, t_s, col_base, s_hi, s_lo, i);
                        cur = nx;
                    } else if (have_nx) {
                        seed_state<kEx>(p, nx, t_s, col_base, s_hi, s_lo, i);
                        cur = nx;
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->s_ready);
                    continue;  // the chunk's output pass is done
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->s_ready);

                if (!(ok = warp_wait_bar(&bars->o_full, gc & 1, limit, abort_flag, p.err))) break;
                tc_fence_after();
                out_pass<2>(tbase + lane_off, col_base, gam, lane, q, r, p.out, r_cur.t0 + cs,
                            row_stride, (size_t)h_cur * head_stride);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->o_free);
            }
            have = have_nx;
        }
        // an S0 load issued and not waited for (the loop left on an abort) lands before the
        // shared memory goes away
        if (threadIdx.x == 0 && s0_issued > nload) {
            int dummy = 0;
            wait_bar(s0_full, (s0_issued - 1) & 1, kDrainLimitNs, &dummy, p.err);
        }
    }

    // the final-state stores this thread issued are complete before the CTA ends
    if (threadIdx.x == 0) bulk_wait_group0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    if (warp == kMmaWarp) {
        __syncwarp();
        tmem_dealloc(tbase, kTmemCols);
    }
}

static_assert(sizeof(Bars) + 3 * sizeof(uint64_t) <= SZ_BAR, "barrier block with the staging barriers");
static_assert(OFF_SLO == OFF_SHI + SZ_T && SZ_T == 2 * 16384 && OFF_SHI % 1024 == 0,
              "the final state's staging: four 16 KiB boxes over S_hi and S_lo, swizzle-aligned");

// The state pool as a TMA map: rows of 128 fp32 (row (slot H + h) 128 + i of slot, head h), boxes
// of 32 columns x 128 rows (a quarter of one state) with the 128-byte swizzle.
typedef CUresult (*EncodeTiledFnM)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_state_map(CUtensorMap *m, float *pool, long long rows) {
    static EncodeTiledFnM fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnM>(f);
    });
    if (!fn || rows <= 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * sizeof(float)};
    const cuuint32_t box[2] = {32, (cuuint32_t)kHeadDim};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, pool, dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Item records: one thread per request computes its rank (request_rank) and writes its geometry
// there, reporting its faults (each request's once) as the one-CTA-per-item kernel does.
__global__ void __launch_bounds__(256) item_records_kernel(const ExtendParams p, ItemRec *recs) {
    pdl_wait();
    pdl_trigger();
    __shared__ int lens[256];
    const int b = blockIdx.x * 256 + threadIdx.x;
    const int t0 = b < p.B ? p.cu_seqlens[b] : 0;
    const int t1 = b < p.B ? p.cu_seqlens[b + 1] : 0;
    const int rank = request_rank(p.cu_seqlens, p.B, b, t1 - t0, lens);
    if (b >= p.B) return;
    ItemRec r{b, t0, 0, p.state_idx[b], 0, 0, 0, 0};
    const int n = t1 - t0;
    if (r.slot < 0 || r.slot >= p.num_slots) {
        atomicOr(p.err, ERR_BIT_SLOT_RANGE);
    } else if (t0 < 0 || t1 < t0 || t1 > p.T || n > p.max_seqlen) {
        atomicOr(p.err, ERR_BIT_SEQLENS);
    } else {
        r.n = n;
        r.flags = kRecValid | (p.prefix_mask[b] ? kRecPrefix : 0);
        // state tracking: the chunk grid restarts at the tracked token (n + 1: none)
        r.sp = n + 1;
        if (p.track_lens != nullptr) {
            const int tl = p.track_lens[b];
            const int ts = p.track_idx[b];
            if (tl >= 0) {
                if (tl > n || ts < 0 || ts >= p.num_slots || ts == r.slot) {
                    atomicOr(p.err, ERR_BIT_TRACK);
                } else {
                    r.sp = tl;
                    r.tslot = ts;
                }
            }
        }
        r.nchunks = r.sp <= n ? (r.sp + C - 1) / C + (n - r.sp + C - 1) / C : (n + C - 1) / C;
    }
    int4 *dst = reinterpret_cast<int4 *>(recs + rank);
    dst[0] = make_int4(r.b, r.t0, r.n, r.slot);
    dst[1] = make_int4(r.sp, r.tslot, r.nchunks, r.flags);
}

}  // namespace

cudaError_t launch_extend_many(const ExtendParams &p, ItemRec *recs, int ctas,
                               cudaStream_t stream) {
    if (ctas <= 0 || p.B <= 0) return cudaSuccess;
    if (recs == nullptr || p.group != 1 || p.seg_len > 0 || p.csplit > 0)
        return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(item_records_kernel, dim3((unsigned)((p.B + 255) / 256)), dim3(256),
                               0, stream, p, recs);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tk, tv, tsm;
    memset(&tq, 0, sizeof(tq));
    memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv));
    memset(&tsm, 0, sizeof(tsm));
    if (p.T > 0) {
        if (!make_token_map_full(&tq, p.q, p.T, p.H) || !make_token_map_full(&tk, p.k, p.T, p.H) ||
            !make_token_map_full(&tv, p.v, p.T, p.H))
            return cudaErrorInvalidValue;
    }
    if (!make_state_map(&tsm, p.pool, (long long)p.num_slots * p.H * kHeadDim))
        return cudaErrorInvalidValue;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static bool configured[64] = {false};
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!configured[dev]) {
            e = cudaFuncSetAttribute(extend_many_kernel<false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(extend_many_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    ExtendParams pw = p;
    pw.recs = recs;
    if (p.track_lens != nullptr || p.out_rs != (long long)p.H * kHeadDim || p.out_hs != kHeadDim)
        return launch_pdl(extend_many_kernel<true>, dim3((unsigned)ctas), dim3(kThreads),
                          kSmemBytes, stream, tq, tk, tv, tsm, pw);
    return launch_pdl(extend_many_kernel<false>, dim3((unsigned)ctas), dim3(kThreads), kSmemBytes,
                      stream, tq, tk, tv, tsm, pw);
}

}  // namespace la
