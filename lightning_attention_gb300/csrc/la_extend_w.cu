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

#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {

namespace {

using namespace sm100;

constexpr int C = 128;              // chunk length in tokens
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kColWarps = kEpiWarps / 4;      // epilogue warps per TMEM lane quarter
constexpr int kKUnits = 16 / kEpiWarps;       // lambda-K units (32 rows x 32 columns) per warp
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr int kThreads = (kEpiWarps + 2) * 32;
// Two warps per lane quarter: each takes 32 of every 64 value columns in the state and output
// passes, so a CTA that covers one 64-column half of the values (nv = 64) still splits evenly.
static_assert(kColWarps == 2, "epilogue warps: 8");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_A = 0;        // 128 columns: Q K^T (fp32), then P (bf16 hi + lo pairs)
constexpr uint32_t TM_OI = 128;     // 128 columns: Q S
constexpr uint32_t TM_OP = 256;     // 128 columns: P V
constexpr uint32_t TM_S = 384;      // 128 columns: the fp32 master state
// head_dim^-0.5 for head_dim = 128, i.e. 2^-3.5
constexpr float kScale = 0.08838834764831845f;

// Shared memory (offsets from a 1024-byte aligned base).  Every tile is [128][128] 16-bit values
// as two 128-byte-swizzled [128][64] blocks 16 KiB apart.
constexpr uint32_t SZ_T = C * kHeadDim * 2;         // 32 KiB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = SZ_T;                    // K of chunk c at OFF_K + (c & 1) SZ_T
constexpr uint32_t OFF_V = OFF_K + 2 * SZ_T;        // V of the chunk in flight (one buffer)
constexpr uint32_t OFF_KLO = OFF_V + SZ_T;          // lo half of lambda K (bf16)
constexpr uint32_t OFF_SHI = OFF_KLO + SZ_T;
constexpr uint32_t OFF_SLO = OFF_SHI + SZ_T;
// e^{-s m} and e^{-s m} D^-0.5 for m = 0..C: read per element only by the P blocks of steep
// decays (slopes above kRunMaxSlope); every other factor is formed in registers
constexpr uint32_t OFF_TAB = OFF_SLO + SZ_T;
constexpr uint32_t OFF_TABP = OFF_TAB + 544;
constexpr uint32_t OFF_BAR = OFF_TABP + 544;
constexpr uint32_t SZ_BAR = 256;
constexpr uint32_t kSmemBytes = OFF_BAR + SZ_BAR + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(OFF_BAR % 8 == 0, "barrier alignment");
static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_KLO % 1024 == 0 &&
                  OFF_SHI % 1024 == 0 && OFF_SLO % 1024 == 0,
              "operand tiles start on 1024-byte swizzle atoms");

struct Bars {
    uint64_t q_full;      // TMA -> all: Q of the chunk loaded
    uint64_t q_empty;     // MMA -> TMA: MMA1 and MMA2 of the chunk done with Q
    uint64_t k_full[2];   // TMA -> all: K of the chunk loaded
    uint64_t k_empty[2];  // MMA -> TMA: MMA1 and MMA4 of the chunk done with K
    uint64_t v_full;      // TMA -> converters: V of the chunk loaded
    uint64_t v_empty;     // MMA -> TMA: MMA4 and MMA3 of the chunk done with V
    uint64_t a_full;      // MMA1 done
    uint64_t k_ready;     // epilogue warps: their share of lambda K written as hi + lo (8)
    uint64_t p_ready;     // epilogue warps: their P blocks written to TMEM (8)
    uint64_t s_ready;     // epilogue: S_hi/S_lo written, decayed S back in TMEM (8)
    uint64_t o_free;      // epilogue: Oint/Ointra read (8)
    uint64_t u_full;      // MMA4 done: S of the chunk complete (and, by issue order, MMA2)
    uint64_t o_full;      // MMA3 done
    uint64_t drain;       // MMA issuer: all MMAs done
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= SZ_BAR, "barrier block");

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

// All 32 lanes wait (each acquires the barrier); the warp proceeds only if every lane succeeded.
__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int *abort_flag, unsigned int *err) {
    const bool ok = wait_bar(bar, parity, limit_ns, abort_flag, err);
    return __all_sync(0xffffffffu, ok);
}

// Descriptor offsets (16-byte units) of the kk-th 16-deep slice of the contraction: K-major tiles
// are two 64-column blocks 16 KiB apart, each slice 32 bytes into the 128-byte row; MN-major
// tiles advance 16 rows (2 KiB) per slice.
__device__ __forceinline__ uint64_t kofs(int kk) {
    return (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2);
}
__device__ __forceinline__ uint64_t mnofs(int kk) { return (uint64_t)(kk * 128); }

// D[tmem] (+)= A[tmem] * B[smem], 16-bit operands (the type is in idesc), fp32 accumulate; issued
// by one thread.  A is M = 128 lanes by K = 16 values, two values per 32-bit column (even index in
// the low half).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-collective TMEM store of 16 consecutive 32-bit columns per lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// 32 state columns (64 atom + 32 sub .. + 31) of row `row` as bf16 hi and lo into the [128][128]
// MN-major operand tiles.
__device__ __forceinline__ void store_state_split(uint8_t *s_hi, uint8_t *s_lo, int row, int atom,
                                                  int sub, const float *S) {
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = S[k4 * 8 + 2 * e], b = S[k4 * 8 + 2 * e + 1];
            const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
            const float2 hf = __bfloat1622float2(h);
            hi[e] = *reinterpret_cast<const uint32_t *>(&h);
            lo[e] = pack_bf16x2(a - hf.x, b - hf.y);
        }
        const int off = atom * 16384 + row * 128 + (((sub * 4 + k4) ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(s_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(s_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// P row segment: 32 columns of block cb of row i, decay-masked and scaled, as a bf16 pair hi + lo
// (16 words each; hi = bf16(x), lo = bf16(x - hi), about 2^-17 together).
// The factor e^{-s (i - j)} D^-0.5 is, for slopes s <= kRunMaxSlope, one table read at j = 32 cb
// followed by a running product with g = e^{s} along the row: this keeps the shared-memory loads,
// which slow down while the MMAs stream their operands, to one per block.  The start value
// e^{-s d} (d <= 127) may then be subnormal, but its error reaches the row only as an absolute
// error below 2^-149 e^{31 s} < 1e-8 of the scale.  Steeper decays read the table per element.
// In the diagonal block the columns past i are zeroed.
constexpr float kRunMaxSlope = 2.5f;

__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16x2(x0, x1);
    lo = pack_bf16x2(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}

__device__ __forceinline__ void p_block(int i, int cb, const uint32_t (&v)[32], const float *tabp,
                                        bool run, float g, float f0, uint32_t (&ph)[16],
                                        uint32_t (&pl)[16]) {
    const int d = i - cb * 32;  // i - j for jj = 0; 0 <= d <= 127 for blocks on or below the diagonal
    if (run) {
        float f = f0;  // e^{-s d} D^-0.5, formed by the caller once per kernel
#pragma unroll
        for (int jj = 0; jj < 32; jj += 2) {
            const float f1 = f * g;
            const float x0 = __uint_as_float(v[jj]) * f, x1 = __uint_as_float(v[jj + 1]) * f1;
            split_bf16x2(jj <= d ? x0 : 0.f, jj + 1 <= d ? x1 : 0.f, ph[jj >> 1], pl[jj >> 1]);
            f = f1 * g;
        }
    } else {
#pragma unroll
        for (int jj = 0; jj < 32; jj += 2) {
            const int d0 = d - jj, d1 = d - jj - 1;
            const float x0 = __uint_as_float(v[jj]) * tabp[max(d0, 0)];
            const float x1 = __uint_as_float(v[jj + 1]) * tabp[max(d1, 0)];
            split_bf16x2(d0 >= 0 ? x0 : 0.f, d1 >= 0 ? x1 : 0.f, ph[jj >> 1], pl[jj >> 1]);
        }
    }
}

// TMEM column of MMA3's A operand for k-step kk (keys 16 kk .. 16 kk + 15): P block kk / 2 sits in
// A block kk / 2, its hi half in the first 16 columns and its lo half in the next 16, one bf16
// pair per column.
__device__ __forceinline__ uint32_t p_col(int kk) { return (uint32_t)(32 * (kk >> 1) + 8 * (kk & 1)); }

// This thread's share of a state (row i, columns col0 .. col0 + 31) into pool slot `slot`.
__device__ __forceinline__ void store_state_row(float *pool, int slot, int H, int h, int i,
                                                int col0, const float *S) {
    float *dst = pool + (((size_t)slot * H + h) * kHeadDim + i) * kHeadDim + (size_t)col0;
#pragma unroll
    for (int x = 0; x < 8; ++x)
        *reinterpret_cast<float4 *>(dst + 4 * x) =
            make_float4(S[4 * x], S[4 * x + 1], S[4 * x + 2], S[4 * x + 3]);
}

// Length of the chunk that starts at local token cs, with the grid restarted at sp (n + 1: none).
__device__ __forceinline__ int chunk_len(bool ex, int cs, int sp, int n) {
    return min(C, (ex && cs < sp ? min(sp, n) : n) - cs);
}

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
            int k_issued = 0, q_issued = 0, v_issued = 0, ys = 0;
            const int xq = h * kHeadDim;    // query head h in q
            const int xkv = hk * kHeadDim;  // its kv head in k and v
            for (int c = 0; c < nchunks; ++c) {
                const int st = c & 1;
                const int y = t0 + (kEx ? ys : c * C);
                if (kEx) ys += chunk_len(true, ys, sp, n);
                // in the order the buffers free up: K (two stages), then Q after MMA2 of the
                // previous chunk, then V after its MMA3
                if (c >= 2 &&
                    !wait_bar(&bars->k_empty[st], ((c >> 1) - 1) & 1, limit, abort_flag, p.err))
                    break;
                uint8_t *kt = sm + OFF_K + st * SZ_T;
                mbar_arrive_expect_tx(&bars->k_full[st], SZ_T);
                tma_load_2d(kt, &tk, &bars->k_full[st], xkv, y);
                tma_load_2d(kt + 16384, &tk, &bars->k_full[st], xkv + 64, y);
                k_issued = c + 1;
                if (c >= 1 && !wait_bar(&bars->q_empty, (c - 1) & 1, limit, abort_flag, p.err))
                    break;
                mbar_arrive_expect_tx(&bars->q_full, SZ_T);
                tma_load_2d(sm + OFF_Q, &tq, &bars->q_full, xq, y);
                tma_load_2d(sm + OFF_Q + 16384, &tq, &bars->q_full, xq + 64, y);
                q_issued = c + 1;
                if (c >= 1 && !wait_bar(&bars->v_empty, (c - 1) & 1, limit, abort_flag, p.err))
                    break;
                if constexpr (nv == kHeadDim) {
                    mbar_arrive_expect_tx(&bars->v_full, SZ_T);
                    tma_load_2d(sm + OFF_V, &tv, &bars->v_full, xkv, y);
                    tma_load_2d(sm + OFF_V + 16384, &tv, &bars->v_full, xkv + 64, y);
                } else {
                    mbar_arrive_expect_tx(&bars->v_full, SZ_T / 2);
                    tma_load_2d(sm + OFF_V, &tv, &bars->v_full, xkv + c0, y);
                }
                v_issued = c + 1;
            }
            // Copies still in flight must land before the CTA's shared memory goes away.
            int dummy = 0;
            for (int c = (k_issued >= 2 ? k_issued - 2 : 0); c < k_issued; ++c)
                wait_bar(&bars->k_full[c & 1], (c >> 1) & 1, kDrainLimitNs, &dummy, p.err);
            if (q_issued > 0)
                wait_bar(&bars->q_full, (q_issued - 1) & 1, kDrainLimitNs, &dummy, p.err);
            if (v_issued > 0)
                wait_bar(&bars->v_full, (v_issued - 1) & 1, kDrainLimitNs, &dummy, p.err);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idA = idesc_bf16_f32(128, 128, false, false);
            // the products with V or S are nv columns wide
            const uint32_t idI = idesc_bf16_f32(128, nv, false, true);
            const uint32_t idP = idesc_bf16_f32(128, nv, false, true);
            const uint32_t idU = idesc_bf16_f32(128, nv, true, true);
            const uint64_t dQ = sdesc_sw128(s_base + OFF_Q, 16, 1024);
            const uint64_t dK0 = sdesc_sw128(s_base + OFF_K, 16, 1024);
            const uint64_t dKt0 = sdesc_sw128(s_base + OFF_K, 16384, 1024);
            const uint64_t dKlo = sdesc_sw128(s_base + OFF_KLO, 16384, 1024);
            const uint64_t dV = sdesc_sw128(s_base + OFF_V, 16384, 1024);
            const uint64_t stage_step = SZ_T >> 4;
            const uint64_t dHi = sdesc_sw128(s_base + OFF_SHI, 16384, 1024);
            const uint64_t dLo = sdesc_sw128(s_base + OFF_SLO, 16384, 1024);
            auto issue_qk = [&](int c) -> bool {
                const int st = c & 1;
                if (!wait_bar(&bars->q_full, c & 1, limit, abort_flag, p.err) ||
                    !wait_bar(&bars->k_full[st], (c >> 1) & 1, limit, abort_flag, p.err))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + TM_A, dQ + kofs(kk), dK0 + st * stage_step + kofs(kk), idA,
                             kk > 0);
                mma_commit(&bars->a_full);
                return true;
            };
            bool ok = true;
            if (nchunks > 0) ok = issue_qk(0);
            for (int c = 0; c < nchunks && ok; ++c) {
                const int st = c & 1;
                // Oint = Q S_{c-1}: needs the previous state and the previous outputs read
                if (!wait_bar(&bars->s_ready, c & 1, limit, abort_flag, p.err) ||
                    (c >= 1 && !wait_bar(&bars->o_free, (c - 1) & 1, limit, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + TM_OI, dQ + kofs(kk), dHi + mnofs(kk), idI, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + TM_OI, dQ + kofs(kk), dLo + mnofs(kk), idI, 1);
                mma_commit(&bars->q_empty);
                // S += (lambda K)^T V once K is scaled and V converted: it runs while P is built
                if (!wait_bar(&bars->k_ready, c & 1, limit, abort_flag, p.err) ||
                    !wait_bar(&bars->v_full, c & 1, limit, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + TM_S, dKt0 + st * stage_step + mnofs(kk), dV + mnofs(kk), idU,
                             1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + TM_S, dKlo + mnofs(kk), dV + mnofs(kk), idU, 1);
                mma_commit(&bars->u_full);
                mma_commit(&bars->k_empty[st]);
                // Ointra = P_hi V + P_lo V once P is in TMEM: it runs while the epilogue does the
                // state pass
                if (!wait_bar(&bars->p_ready, c & 1, limit, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_f16_tmem_a(tbase + TM_OP, tbase + TM_A + p_col(kk),
                                   dV + mnofs(kk), idP, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_f16_tmem_a(tbase + TM_OP, tbase + TM_A + p_col(kk) + 16u,
                                   dV + mnofs(kk), idP, 1);
                mma_commit(&bars->o_full);
                mma_commit(&bars->v_empty);
                if (c + 1 < nchunks && !(ok = issue_qk(c + 1))) break;
            }
            // Every issued MMA must finish before TMEM is freed.
            mma_commit(&bars->drain);
            int dummy = 0;
            wait_bar(&bars->drain, 0, kDrainLimitNs, &dummy, p.err);
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
            // all units' loads are issued before any is converted, so the warp waits for one
            // shared-memory round trip
            {
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
                    lrow[k] = reinterpret_cast<uint4 *>(sm + OFF_KLO + roff);
                    h4[k] = (u & 1) * 4;
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) kbuf[k][ch] = krow[k][(h4[k] + ch + rr[k]) & 7];
                }
#pragma unroll
                for (int k = 0; k < kKUnits; ++k) {
                    const LamSplitBf lam = r == C ? lam_full[k]
                                                  : lam_split_bf16(rr[k] < r ? expf(-slope * (float)(r - 1 - rr[k]))
                                                                             : 0.f);
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint4 hi, lo;
                        bf16x8_lam_hilo_bf16(kbuf[k][ch], lam, hi, lo);
                        krow[k][(h4[k] + ch + rr[k]) & 7] = hi;
                        lrow[k][(h4[k] + ch + rr[k]) & 7] = lo;
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->k_ready);
            {
                // ---- P = A o Dm D^-0.5 into TMEM: block cb (keys 32 cb .. 32 cb + 31) goes as a
                // bf16 pair hi + lo over its own A block's 32 columns, so a warp only overwrites
                // what it has read itself; blocks above the diagonal are zeroed
                const uint32_t ta = tbase + lane_off + TM_A;
#pragma unroll 1
                for (int cb = pb0; cb < pb1; ++cb) {
                    uint32_t ph[16], pl[16];
                    uint32_t va[32];
                    tmem_ld32(ta + (uint32_t)cb * 32u, va);
                    tmem_ld_wait_regs(va);
                    p_block(i, cb, va, tabp, run, grow, cb == pb0 ? f_p0 : f_p1, ph, pl);
                    tmem_st16(ta + (uint32_t)cb * 32u, ph);
                    tmem_st16(ta + (uint32_t)cb * 32u + 16u, pl);
                }
                if (zb0 < zb1) {
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) pk[x] = 0u;
                    for (int cb = zb0; cb < zb1; ++cb) {
                        tmem_st16(ta + (uint32_t)cb * 32u, pk);
                        tmem_st16(ta + (uint32_t)cb * 32u + 16u, pk);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_ready);
            }

            // ---- state: S_c is in TMEM once MMA4 is done; hi/lo copy for MMA2_{c+1}, then
            // e^{-s r_{c+1}} S_c back for MMA4_{c+1}
            if (!(ok = warp_wait_bar(&bars->u_full, c & 1, limit, abort_flag, p.err))) break;
            tc_fence_after();
            {
                const int r_next = c + 1 < nchunks ? chunk_len(kEx, cs + r, sp, n) : 0;
                const float dn = c + 1 >= nchunks ? 1.f
                                 : r_next == C   ? dn_full
                                                 : expf(-slope * (float)r_next);
#pragma unroll 1
                for (int sub = 0; sub < nsubs; ++sub) {
                    const int col0 = col_base + sub * 32;
                    const uint32_t t_s = tbase + lane_off + TM_S + (uint32_t)col0;
                    uint32_t w[32];
                    tmem_ld32(t_s, w);
                    tmem_ld_wait_regs(w);
                    float S[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        S[x] = __uint_as_float(w[x]);
                        w[x] = __float_as_uint(S[x] * dn);
                    }
                    tmem_st32(t_s, w);
                    store_state_split(s_hi, s_lo, i, col0 >> 6, (col0 >> 5) & 1, S);
                    if (kEx && cs + r == sp)
                        store_state_row(p.pool, p.track_idx[b], H, h, i, c0 + col0, S);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_ready);

            // ---- out: o = gamma D^-0.5 Oint + Ointra -> bf16, 32 columns at a time
            if (!(ok = warp_wait_bar(&bars->o_full, c & 1, limit, abort_flag, p.err))) break;
            tc_fence_after();
#pragma unroll 1
            for (int sub = 0; sub < nsubs; ++sub) {
                const int col0 = col_base + sub * 32;
                uint32_t vi[32], vp[32];
                tmem_ld32(tbase + lane_off + TM_OI + (uint32_t)col0, vi);
                tmem_ld32(tbase + lane_off + TM_OP + (uint32_t)col0, vp);
                tmem_ld_wait_regs2(vi, vp);
                uint4 ch[4];
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int x = k4 * 8 + 2 * e;
                        w[e] = pack_bf16x2(
                            fmaf(gam, __uint_as_float(vi[x]), __uint_as_float(vp[x])),
                            fmaf(gam, __uint_as_float(vi[x + 1]), __uint_as_float(vp[x + 1])));
                    }
                    ch[k4] = make_uint4(w[0], w[1], w[2], w[3]);
                }
                // 4x4 transpose of 16-byte chunks within each group of 4 lanes (two butterfly
                // steps), so that store k writes row 4*(lane/4) + k of the group as one
                // contiguous 64-byte segment per group.
                const int pq = lane & 3;
                {
                    const bool lo2 = pq < 2;
                    uint4 sa = lo2 ? ch[2] : ch[0], sb = lo2 ? ch[3] : ch[1];
                    uint4 ra, rb;
                    ra.x = __shfl_xor_sync(0xffffffffu, sa.x, 2);
                    ra.y = __shfl_xor_sync(0xffffffffu, sa.y, 2);
                    ra.z = __shfl_xor_sync(0xffffffffu, sa.z, 2);
                    ra.w = __shfl_xor_sync(0xffffffffu, sa.w, 2);
                    rb.x = __shfl_xor_sync(0xffffffffu, sb.x, 2);
                    rb.y = __shfl_xor_sync(0xffffffffu, sb.y, 2);
                    rb.z = __shfl_xor_sync(0xffffffffu, sb.z, 2);
                    rb.w = __shfl_xor_sync(0xffffffffu, sb.w, 2);
                    if (lo2) { ch[2] = ra; ch[3] = rb; } else { ch[0] = ra; ch[1] = rb; }
                }
                {
                    const bool even = (pq & 1) == 0;
                    uint4 sa = even ? ch[1] : ch[0], sb = even ? ch[3] : ch[2];
                    uint4 ra, rb;
                    ra.x = __shfl_xor_sync(0xffffffffu, sa.x, 1);
                    ra.y = __shfl_xor_sync(0xffffffffu, sa.y, 1);
                    ra.z = __shfl_xor_sync(0xffffffffu, sa.z, 1);
                    ra.w = __shfl_xor_sync(0xffffffffu, sa.w, 1);
                    rb.x = __shfl_xor_sync(0xffffffffu, sb.x, 1);
                    rb.y = __shfl_xor_sync(0xffffffffu, sb.y, 1);
                    rb.z = __shfl_xor_sync(0xffffffffu, sb.z, 1);
                    rb.w = __shfl_xor_sync(0xffffffffu, sb.w, 1);
                    if (even) { ch[1] = ra; ch[3] = rb; } else { ch[0] = ra; ch[2] = rb; }
                }
                // lane (4 g + pq) now holds chunk pq of rows 4 g .. 4 g + 3 of its warp's rows
                const int rbase = q * 32 + (lane & ~3);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int row = rbase + k;
                    if (row < r) {
                        __nv_bfloat16 *dst = p.out + (size_t)(t0 + cs + row) * row_stride +
                                             (size_t)h * head_stride + c0 + col0 + pq * 8;
                        *reinterpret_cast<uint4 *>(dst) = ch[k];
                    }
                }
            }
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
