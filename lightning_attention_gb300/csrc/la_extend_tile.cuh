// la_extend_tile.cuh -- what the extend kernels share: the chunk length and warp roles, the
// tensor-memory and shared-memory layout of a CTA, its mbarriers with their bounded waits, the
// operand descriptors, and the epilogue warps' per-chunk passes (lambda K, P, state, output).
//
// Method: page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section
// "独立参考实现：逐 token 递推公式", in the chunked form that la_extend_w.cu states: per chunk of
// r tokens with local indices i, j and S the state before it,
//   o_i    = D^-0.5 gamma_i (Q S)_i + ((Q K^T o Dm) D^-0.5 V)_i,   gamma_i = e^{-s (i+1)},
//   S_next = e^{-s r} S + K^T diag(lambda) V,                       lambda_j = e^{-s (r-1-j)}.
// Two kernels use it: one CTA per (request, head) (la_extend_w.cu) and the persistent grid that
// works through batches of more than one wave (la_extend_many.cu).
#pragma once

#include <cuda.h>

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
// error below 2^-149 e^{31 s} < 1e-8 of the scale.  Steeper decays take the factor per element,
// from the table (kTab) or from the exponential.
// In the diagonal block the columns past i are zeroed.
constexpr float kRunMaxSlope = 2.5f;

__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16x2(x0, x1);
    lo = pack_bf16x2(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}

template <bool kTab>
__device__ __forceinline__ void p_block(int i, int cb, const uint32_t (&v)[32], const float *tabp,
                                        float slope, bool run, float g, float f0,
                                        uint32_t (&ph)[16], uint32_t (&pl)[16]) {
    const int d = i - cb * 32;  // i - j for jj = 0; 0 <= d <= 127 for blocks on or below the diagonal
    if (run) {
        float f = f0;  // e^{-s d} D^-0.5, formed by the caller once per (request, head)
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
            float e0, e1;
            if constexpr (kTab) {
                e0 = tabp[max(d0, 0)];
                e1 = tabp[max(d1, 0)];
            } else {
                e0 = expf(-slope * (float)max(d0, 0)) * kScale;
                e1 = expf(-slope * (float)max(d1, 0)) * kScale;
            }
            const float x0 = __uint_as_float(v[jj]) * e0;
            const float x1 = __uint_as_float(v[jj + 1]) * e1;
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

// Chunks whose K, Q and V loads the TMA producer has issued.
struct Issued {
    int k, q, v;
};

// The TMA producer's loads of chunk c of the stream, token row y (query head columns xq .., kv
// head columns xkv .., value columns c0 .. c0 + nv - 1 of it): in the order the buffers free up,
// K into stage c & 1 once MMA1 and MMA4 of chunk c - 2 are done with it, then Q once MMA2 of
// chunk c - 1 is, then V once MMA3 of chunk c - 1 is.  False: a wait gave up.
template <int nv>
__device__ __forceinline__ bool produce_chunk(Bars *bars, uint8_t *sm, const CUtensorMap &tq,
                                              const CUtensorMap &tk, const CUtensorMap &tv, int c,
                                              int y, int xq, int xkv, int c0, uint64_t limit,
                                              volatile int *abort_flag, unsigned int *err,
                                              Issued &is) {
    const int st = c & 1;
    if (c >= 2 && !wait_bar(&bars->k_empty[st], ((c >> 1) - 1) & 1, limit, abort_flag, err))
        return false;
    uint8_t *kt = sm + OFF_K + st * SZ_T;
    mbar_arrive_expect_tx(&bars->k_full[st], SZ_T);
    tma_load_2d(kt, &tk, &bars->k_full[st], xkv, y);
    tma_load_2d(kt + 16384, &tk, &bars->k_full[st], xkv + 64, y);
    is.k = c + 1;
    if (c >= 1 && !wait_bar(&bars->q_empty, (c - 1) & 1, limit, abort_flag, err)) return false;
    mbar_arrive_expect_tx(&bars->q_full, SZ_T);
    tma_load_2d(sm + OFF_Q, &tq, &bars->q_full, xq, y);
    tma_load_2d(sm + OFF_Q + 16384, &tq, &bars->q_full, xq + 64, y);
    is.q = c + 1;
    if (c >= 1 && !wait_bar(&bars->v_empty, (c - 1) & 1, limit, abort_flag, err)) return false;
    if constexpr (nv == kHeadDim) {
        (void)c0;
        mbar_arrive_expect_tx(&bars->v_full, SZ_T);
        tma_load_2d(sm + OFF_V, &tv, &bars->v_full, xkv, y);
        tma_load_2d(sm + OFF_V + 16384, &tv, &bars->v_full, xkv + 64, y);
    } else {
        mbar_arrive_expect_tx(&bars->v_full, SZ_T / 2);
        tma_load_2d(sm + OFF_V, &tv, &bars->v_full, xkv + c0, y);
    }
    is.v = c + 1;
    return true;
}

// Copies still in flight must land before the CTA's shared memory goes away.
__device__ __forceinline__ void produce_drain(Bars *bars, const Issued &is, unsigned int *err) {
    int dummy = 0;
    for (int c = (is.k >= 2 ? is.k - 2 : 0); c < is.k; ++c)
        wait_bar(&bars->k_full[c & 1], (c >> 1) & 1, kDrainLimitNs, &dummy, err);
    if (is.q > 0) wait_bar(&bars->q_full, (is.q - 1) & 1, kDrainLimitNs, &dummy, err);
    if (is.v > 0) wait_bar(&bars->v_full, (is.v - 1) & 1, kDrainLimitNs, &dummy, err);
}

// The MMA issuer's loop (one thread) over a stream of nchunks chunks, nv value columns: for chunk c,
// MMA2 (Q S_hi + Q S_lo -> Oint) once the state pass of c - 1 and the output pass of c - 1 are
// done, MMA4 (S += (lambda K)_hi^T V + (lambda K)_lo^T V) once lambda K and V are in, MMA3 (P_hi V
// + P_lo V -> Ointra) once P is in TMEM, then MMA1 of c + 1 (Q K^T -> A).  Barrier parities count
// chunks of the stream.  On return every issued MMA has completed (or the drain wait gave up).
template <int nv>
__device__ __forceinline__ void mma_loop(Bars *bars, uint32_t tbase, uint32_t s_base, int nchunks,
                                         uint64_t limit, volatile int *abort_flag,
                                         unsigned int *err) {
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
        if (!wait_bar(&bars->q_full, c & 1, limit, abort_flag, err) ||
            !wait_bar(&bars->k_full[st], (c >> 1) & 1, limit, abort_flag, err))
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
        if (!wait_bar(&bars->s_ready, c & 1, limit, abort_flag, err) ||
            (c >= 1 && !wait_bar(&bars->o_free, (c - 1) & 1, limit, abort_flag, err))) {
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
        if (!wait_bar(&bars->k_ready, c & 1, limit, abort_flag, err) ||
            !wait_bar(&bars->v_full, c & 1, limit, abort_flag, err)) {
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
        if (!wait_bar(&bars->p_ready, c & 1, limit, abort_flag, err)) {
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
    wait_bar(&bars->drain, 0, kDrainLimitNs, &dummy, err);
}

// ---------------------------------------------------------------------------------------------
// The epilogue warps' per-chunk passes.  Warp w owns TMEM lane quarter q = w % 4 (rows i = 32 q +
// lane of A, P, Oint, Ointra and of the state) and column slot cw = w / 4 of the state and output
// passes; nsubs is the number of 32-column parts of its slot (2 at 128 value columns, 1 at 64).

// Lambda K of the chunk in K stage st as a bf16 pair: hi in place in the K tile, lo into its own
// buffer, for this warp's kKUnits units of 32 rows x 32 columns (unit u: rows 32 (u / 4) .., column
// quarter u % 4).  lam_full holds the units' row factors of a full chunk; a ragged chunk of r
// tokens forms its own (rows past r scale to zero).  All units' loads are issued before any is
// converted, so the warp waits for one shared-memory round trip.
__device__ __forceinline__ void lamk_pass(uint8_t *sm, int st, int ku0, int lane, int r,
                                          float slope, const LamSplitBf (&lam_full)[kKUnits]) {
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

// P = A o Dm D^-0.5 into TMEM (ta: this warp's lanes of the A block): block cb (keys 32 cb ..
// 32 cb + 31) of this warp's blocks pb0 .. pb1 - 1 goes as a bf16 pair hi + lo over its own A
// block's 32 columns, so a warp only overwrites what it has read itself; blocks zb0 .. zb1 - 1
// above the diagonal are zeroed.  f_p0, f_p1: start factors of blocks pb0 and pb0 + 1.
template <bool kTab>
__device__ __forceinline__ void p_pass(uint32_t ta, int i, int pb0, int pb1, int zb0, int zb1,
                                       const float *tabp, float slope, bool run, float grow,
                                       float f_p0, float f_p1) {
#pragma unroll 1
    for (int cb = pb0; cb < pb1; ++cb) {
        uint32_t ph[16], pl[16];
        uint32_t va[32];
        tmem_ld32(ta + (uint32_t)cb * 32u, va);
        tmem_ld_wait_regs(va);
        p_block<kTab>(i, cb, va, tabp, slope, run, grow, cb == pb0 ? f_p0 : f_p1, ph, pl);
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
}

// State pass: S of the chunk (t_s: this warp's lanes of the state columns) as a bf16 pair into
// the MMA2 operand tiles, and dn S back into TMEM for the next chunk's MMA4.  With kEx and snap,
// the state is also stored into slot tslot of the pool (a tracking snapshot).
template <bool kEx, int nsubs>
__device__ __forceinline__ void state_pass(uint32_t t_s, int col_base, uint8_t *s_hi,
                                           uint8_t *s_lo, int i, float dn, bool snap,
                                           float *pool, int tslot, int H, int h, int c0) {
#pragma unroll 1
    for (int sub = 0; sub < nsubs; ++sub) {
        const int col0 = col_base + sub * 32;
        uint32_t w[32];
        tmem_ld32(t_s + (uint32_t)col0, w);
        tmem_ld_wait_regs(w);
        float S[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) {
            S[x] = __uint_as_float(w[x]);
            w[x] = __float_as_uint(S[x] * dn);
        }
        tmem_st32(t_s + (uint32_t)col0, w);
        store_state_split(s_hi, s_lo, i, col0 >> 6, (col0 >> 5) & 1, S);
        if (kEx && snap) store_state_row(pool, tslot, H, h, i, c0 + col0, S);
    }
    tmem_st_wait();
}

// Output pass: o = gam Oint + Ointra (gam = gamma_i D^-0.5) -> bf16, 32 columns at a time (t_l:
// this warp's lanes), rows 0 .. r - 1 of the chunk; row x of column j goes to
// out[(t_row + x) row_stride + col_off + j].
template <int nsubs>
__device__ __forceinline__ void out_pass(uint32_t t_l, int col_base, float gam, int lane, int q,
                                         int r, __nv_bfloat16 *out, int t_row, size_t row_stride,
                                         size_t col_off) {
#pragma unroll 1
    for (int sub = 0; sub < nsubs; ++sub) {
        const int col0 = col_base + sub * 32;
        uint32_t vi[32], vp[32];
        tmem_ld32(t_l + TM_OI + (uint32_t)col0, vi);
        tmem_ld32(t_l + TM_OP + (uint32_t)col0, vp);
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
        // 4x4 transpose of 16-byte chunks within each group of 4 lanes (two butterfly steps), so
        // that store k writes row 4*(lane/4) + k of the group as one contiguous 64-byte segment
        // per group.
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
                __nv_bfloat16 *dst =
                    out + (size_t)(t_row + row) * row_stride + col_off + col0 + pq * 8;
                *reinterpret_cast<uint4 *>(dst) = ch[k];
            }
        }
    }
}

}  // namespace

}  // namespace la
