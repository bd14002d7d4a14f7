// la_recurrent.cu -- token-serial seg_la kernels: one-token decode, chain and tree verify.
//
// Method: page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section
// "独立参考实现：逐 token 递推公式":  S_t = S_{t-1} * exp(-slope_h) + outer(k_t, v_t),
// o_t = (q_t @ S_t) * D^-0.5.  Chain verify follows the same page's section "生产环境不支持",
// item 3 (every draft token continues from the previous position); tree verify follows its
// section "Next Work", item 2 (each draft token forks from the state saved for its parent).
//
// These paths are HBM-bound: per (request, head) the 128 x 128 fp32 state (64 KiB) is read once,
// updated token by token in registers, and written once (decode: back to the pool; verify: once
// per draft token into the intermediate-state buffer).  Design for GB300:
//   * one CTA of 256 threads per (request, head); warp w owns state rows [16w, 16w+16), lane l
//     owns columns [4l, 4l+4), so every state access is a 16-byte vector load/store and a warp
//     touches 512 contiguous bytes of a row -- fully coalesced;
//   * all 16 row loads of a thread are issued back to back before any arithmetic (64 KiB in
//     flight per CTA), with evict-first cache hints since the state is touched exactly once;
//   * the readout q @ S contracts over rows, i.e. across the 8 warps: each thread accumulates its
//     16-row partial sum in registers and the 8 partials meet in shared memory (double-buffered,
//     so one __syncthreads per token suffices);
//   * the decay is applied and the outer product added with one FMA per state element.
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kHeadDim / kWarps;  // 16
// head_dim^-0.5 for head_dim = 128, i.e. 2^-3.5
constexpr float kScale = 0.08838834764831845f;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
    f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
    f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(const RecurParams p) {
    pdl_wait();
    pdl_trigger();
    const int H = p.H;
    const int b = blockIdx.x / H;
    const int h = blockIdx.x - b * H;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row0 = warp * kRowsPerWarp;
    const int col = lane * 4;

    __shared__ __align__(16) float red[2][kWarps][kHeadDim];

    const int slot = p.state_idx[b];
    if (slot < 0 || slot >= p.num_slots) {
        if (threadIdx.x == 0) atomicOr(p.err, ERR_BIT_SLOT_RANGE);
        return;
    }
    float *state = p.pool + ((size_t)slot * H + h) * (size_t)(kHeadDim * kHeadDim);

    const int t_begin = MODE == RECUR_DECODE ? b : b * p.N;
    const int n = MODE == RECUR_DECODE ? 1 : p.N;
    // Tree: the states that a later token forks from (bit t) are stored with the default cache
    // policy so that the fork reloads them from L2; every other intermediate state is streamed.
    unsigned long long reused = 0ull;
    if (MODE == RECUR_TREE) {
        // parents must point backwards; checked up front so that a bad tree writes nothing
        bool bad = false;
        for (int t = 0; t < n; ++t) {
            const int par = p.parents[(size_t)b * p.N + t];
            bad |= par < -1 || par >= t;
            if (par >= 0 && par != t - 1 && par < 64) reused |= 1ull << par;
        }
        if (bad) {
            if (threadIdx.x == 0) atomicOr(p.err, ERR_BIT_PARENTS);
            return;
        }
    }

    float4 s[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
        s[r] = __ldcs(reinterpret_cast<const float4 *>(state + (size_t)(row0 + r) * kHeadDim + col));

    const float decay = expf(-p.slopes[h]);
    const size_t row_stride = (size_t)H * kHeadDim;

    for (int t = 0; t < n; ++t) {
        if (MODE == RECUR_TREE) {
            // Fork: unless the parent is the previous token (state already in registers), reload
            // the parent's state -- the pool slot for the root, else the intermediate state this
            // thread itself stored for the parent (same elements, so no cross-thread ordering).
            const int par = p.parents[(size_t)b * p.N + t];
            if (par != t - 1) {
                const float *src =
                    par < 0 ? state
                            : p.inter + (((size_t)b * p.N + par) * H + h) *
                                            (size_t)(kHeadDim * kHeadDim);
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r)
                    s[r] = *reinterpret_cast<const float4 *>(src + (size_t)(row0 + r) * kHeadDim +
                                                             col);
            }
        }
        const size_t tok = (size_t)(t_begin + t) * row_stride + (size_t)h * kHeadDim;
        // this warp's 16 k and q entries (same address across the warp: a broadcast) and this
        // lane's 4 v entries
        const uint4 *kp = reinterpret_cast<const uint4 *>(p.k + tok + row0);
        const uint4 *qp = reinterpret_cast<const uint4 *>(p.q + tok + row0);
        const uint2 vv = *reinterpret_cast<const uint2 *>(p.v + tok + col);
        float kf[16], qf[16];
        unpack8(kp[0], kf);
        unpack8(kp[1], kf + 8);
        unpack8(qp[0], qf);
        unpack8(qp[1], qf + 8);
        const float v0 = bf_lo(vv.x), v1 = bf_hi(vv.x), v2 = bf_lo(vv.y), v3 = bf_hi(vv.y);

        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            // S = S * exp(-slope) + outer(k, v), one FMA per element
            s[r].x = fmaf(kf[r], v0, s[r].x * decay);
            s[r].y = fmaf(kf[r], v1, s[r].y * decay);
            s[r].z = fmaf(kf[r], v2, s[r].z * decay);
            s[r].w = fmaf(kf[r], v3, s[r].w * decay);
            o.x = fmaf(qf[r], s[r].x, o.x);
            o.y = fmaf(qf[r], s[r].y, o.y);
            o.z = fmaf(qf[r], s[r].z, o.z);
            o.w = fmaf(qf[r], s[r].w, o.w);
        }
        if (MODE == RECUR_VERIFY || MODE == RECUR_TREE) {
            float *dst = p.inter + (((size_t)b * p.N + t) * H + h) * (size_t)(kHeadDim * kHeadDim);
            if (MODE == RECUR_TREE && t < 64 && ((reused >> t) & 1ull)) {
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r)
                    *reinterpret_cast<float4 *>(dst + (size_t)(row0 + r) * kHeadDim + col) = s[r];
            } else {
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r)
                    __stcs(reinterpret_cast<float4 *>(dst + (size_t)(row0 + r) * kHeadDim + col),
                           s[r]);
            }
        }
        float(*buf)[kHeadDim] = red[t & 1];
        *reinterpret_cast<float4 *>(&buf[warp][col]) = o;
        __syncthreads();
        if (threadIdx.x < kHeadDim / 2) {
            const int j = threadIdx.x * 2;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                a0 += buf[w][j];
                a1 += buf[w][j + 1];
            }
            *reinterpret_cast<__nv_bfloat162 *>(p.out + tok + j) =
                __floats2bfloat162_rn(a0 * kScale, a1 * kScale);
        }
        // red[t & 1] is rewritten at token t + 2, after every reader has passed the barrier of
        // token t + 1, so one barrier per token is enough.
    }

    if (MODE == RECUR_DECODE) {
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
            __stcs(reinterpret_cast<float4 *>(state + (size_t)(row0 + r) * kHeadDim + col), s[r]);
    }
}

// Grouped-query decode: CTA (b, j) advances the state of kv head j of request b by one token and
// reads it out for the G query heads j G .. j G + G - 1, so each state crosses HBM once however
// many query heads share it.  Thread layout, vector widths and the per-token arithmetic are those
// of recurrent_kernel; the readouts meet in the same double-buffered shared memory, one barrier
// per query head.
__global__ void __launch_bounds__(kThreads) decode_grouped_kernel(const RecurParams p) {
    pdl_wait();
    pdl_trigger();
    const int H = p.H;  // kv heads
    const int G = p.G;
    const int b = blockIdx.x / H;
    const int j = blockIdx.x - b * H;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row0 = warp * kRowsPerWarp;
    const int col = lane * 4;

    __shared__ __align__(16) float red[2][kWarps][kHeadDim];

    const int slot = p.state_idx[b];
    if (slot < 0 || slot >= p.num_slots) {
        if (threadIdx.x == 0) atomicOr(p.err, ERR_BIT_SLOT_RANGE);
        return;
    }
    float *state = p.pool + ((size_t)slot * H + j) * (size_t)(kHeadDim * kHeadDim);
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
        s[r] = __ldcs(reinterpret_cast<const float4 *>(state + (size_t)(row0 + r) * kHeadDim + col));

    const float decay = expf(-p.slopes[j]);
    const size_t kv = (size_t)b * H * kHeadDim + (size_t)j * kHeadDim;
    const uint4 *kp = reinterpret_cast<const uint4 *>(p.k + kv + row0);
    const uint2 vv = *reinterpret_cast<const uint2 *>(p.v + kv + col);
    float kf[16];
    unpack8(kp[0], kf);
    unpack8(kp[1], kf + 8);
    const float v0 = bf_lo(vv.x), v1 = bf_hi(vv.x), v2 = bf_lo(vv.y), v3 = bf_hi(vv.y);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        // S = S * exp(-slope_j) + outer(k, v), once for the whole group
        s[r].x = fmaf(kf[r], v0, s[r].x * decay);
        s[r].y = fmaf(kf[r], v1, s[r].y * decay);
        s[r].z = fmaf(kf[r], v2, s[r].z * decay);
        s[r].w = fmaf(kf[r], v3, s[r].w * decay);
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
        __stcs(reinterpret_cast<float4 *>(state + (size_t)(row0 + r) * kHeadDim + col), s[r]);

    const size_t q_row = (size_t)H * G * kHeadDim;
    for (int g = 0; g < G; ++g) {
        const size_t qo = (size_t)b * q_row + (size_t)(j * G + g) * kHeadDim;
        const uint4 *qp = reinterpret_cast<const uint4 *>(p.q + qo + row0);
        float qf[16];
        unpack8(qp[0], qf);
        unpack8(qp[1], qf + 8);
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            o.x = fmaf(qf[r], s[r].x, o.x);
            o.y = fmaf(qf[r], s[r].y, o.y);
            o.z = fmaf(qf[r], s[r].z, o.z);
            o.w = fmaf(qf[r], s[r].w, o.w);
        }
        float(*buf)[kHeadDim] = red[g & 1];
        *reinterpret_cast<float4 *>(&buf[warp][col]) = o;
        __syncthreads();
        if (threadIdx.x < kHeadDim / 2) {
            const int jj = threadIdx.x * 2;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                a0 += buf[w][jj];
                a1 += buf[w][jj + 1];
            }
            *reinterpret_cast<__nv_bfloat162 *>(p.out + qo + jj) =
                __floats2bfloat162_rn(a0 * kScale, a1 * kScale);
        }
        // red[g & 1] is rewritten at query head g + 2, after every reader of head g has passed
        // the barrier of head g + 1
    }
}

// One CTA of 256 threads per (request, head): a 64 KiB fp32 copy with 16-byte accesses.
__global__ void __launch_bounds__(kThreads) commit_kernel(const CommitParams p) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x / p.H;
    const int h = blockIdx.x - b * p.H;
    const int slot = p.state_idx[b];
    const int a = p.accept_idx[b];
    if (slot < 0 || slot >= p.num_slots) {
        if (threadIdx.x == 0) atomicOr(p.err, ERR_BIT_SLOT_RANGE);
        return;
    }
    if (a < -1 || a >= p.N) {
        if (threadIdx.x == 0) atomicOr(p.err, ERR_BIT_ACCEPT);
        return;
    }
    if (a < 0) return;  // nothing accepted: the slot keeps its state
    const float4 *src = reinterpret_cast<const float4 *>(
        p.inter + (((size_t)b * p.N + a) * p.H + h) * (size_t)(kHeadDim * kHeadDim));
    float4 *dst =
        reinterpret_cast<float4 *>(p.pool + ((size_t)slot * p.H + h) * (size_t)(kHeadDim * kHeadDim));
    constexpr int kVec = kHeadDim * kHeadDim / 4;
    float4 buf[kVec / kThreads];
#pragma unroll
    for (int x = 0; x < kVec / kThreads; ++x) buf[x] = __ldcs(src + threadIdx.x + x * kThreads);
#pragma unroll
    for (int x = 0; x < kVec / kThreads; ++x) dst[threadIdx.x + x * kThreads] = buf[x];
}

}  // namespace

cudaError_t launch_commit(const CommitParams &p, cudaStream_t stream) {
    const long long blocks = (long long)p.B * p.H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_pdl(commit_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p);
}

cudaError_t launch_decode_grouped(const RecurParams &p, cudaStream_t stream) {
    const long long blocks = (long long)p.B * p.H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_pdl(decode_grouped_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p);
}

cudaError_t launch_recurrent(RecurMode mode, const RecurParams &p, cudaStream_t stream) {
    const long long blocks = (long long)p.B * p.H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)blocks), block(kThreads);
    switch (mode) {
        case RECUR_DECODE:
            return launch_pdl(recurrent_kernel<RECUR_DECODE>, grid, block, 0, stream, p);
        case RECUR_VERIFY:
            return launch_pdl(recurrent_kernel<RECUR_VERIFY>, grid, block, 0, stream, p);
        case RECUR_TREE:
            return launch_pdl(recurrent_kernel<RECUR_TREE>, grid, block, 0, stream, p);
    }
    return cudaErrorInvalidValue;
}

}  // namespace la
