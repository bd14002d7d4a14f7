// la_internal.h -- declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace la {

// Programmatic dependent launch.  Every kernel of the library is launched with programmatic
// stream serialization, so that it may be scheduled while the previous kernel on the stream
// drains; it calls pdl_wait() before its first global-memory access (which returns once that
// kernel has completed and its writes are visible, at once when there is none in flight) and
// pdl_trigger() right after, so that the next kernel may be scheduled in turn.  A predecessor
// that never triggers (any kernel outside the library) is simply waited for, as without the
// attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Rank of request b (length lb) in decreasing length order: the number of the B requests that
// are longer, or as long with a smaller index.  A strict total order, so the ranks are a
// permutation even for inconsistent cu_seqlens (which the extend kernels report).  Every thread
// of the 256-thread block calls it (b past B too); the lengths are staged through `lens` 256 at
// a time.
__device__ __forceinline__ int request_rank(const int32_t *cu_seqlens, int B, int b, int lb,
                                            int (&lens)[256]) {
    int rank = 0;
    for (int u0 = 0; u0 < B; u0 += 256) {
        __syncthreads();
        const int u = u0 + threadIdx.x;
        lens[threadIdx.x] = u < B ? cu_seqlens[u + 1] - cu_seqlens[u] : 0;
        __syncthreads();
        const int m = B - u0 < 256 ? B - u0 : 256;
        for (int x = 0; x < m; ++x) {
            const int lu = lens[x];
            rank += (lu > lb) || (lu == lb && u0 + x < b);
        }
    }
    return rank;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Bits of the per-device error word (see la_api.cu).
enum : unsigned int {
    ERR_BIT_TIMEOUT = 1u,       // a bounded device wait ran out
    ERR_BIT_SLOT_RANGE = 2u,    // state_idx entry outside [0, num_slots)
    ERR_BIT_SEQLENS = 4u,       // cu_seqlens decreasing or past T
    ERR_BIT_PARENTS = 8u,       // tree-verify parent index outside [-1, t-1]
    ERR_BIT_ACCEPT = 16u,       // commit index outside [-1, N-1]
    ERR_BIT_TRACK = 32u,        // track length outside [-1, n] or bad track slot
};

constexpr int kHeadDim = 128;

// Recurrent (token-serial) kernels: decode, chain and tree verify.
enum RecurMode : int { RECUR_DECODE = 0, RECUR_VERIFY = 1, RECUR_TREE = 3 };

struct RecurParams {
    const __nv_bfloat16 *q, *k, *v;
    const float *slopes;
    float *pool;                 // [num_slots][H][D][D]
    const int32_t *state_idx;    // [B]
    float *inter;                // [B][N][H][D][D] (verify)
    const int32_t *parents;      // [B][N] (tree verify)
    __nv_bfloat16 *out;
    unsigned int *err;           // device error word
    int B, H, N, num_slots;      // H: heads of k, v, slopes and the states
    int G;                       // query heads per state (grouped decode; 1 otherwise): q and out
                                 // have H * G heads, query head h reads state h / G
};

cudaError_t launch_recurrent(RecurMode mode, const RecurParams &p, cudaStream_t stream);
// Grouped-query decode: one CTA per (request, kv head) advances the state once and reads it out
// for each of its p.G query heads.
cudaError_t launch_decode_grouped(const RecurParams &p, cudaStream_t stream);

// Accepted-state commit: pool[state_idx[b]] = inter[b][accept_idx[b]] (all heads) when
// accept_idx[b] >= 0.
struct CommitParams {
    const float *inter;          // [B][N][H][D][D]
    const int32_t *accept_idx;   // [B]
    float *pool;
    const int32_t *state_idx;
    unsigned int *err;
    int B, N, H, num_slots;
};
cudaError_t launch_commit(const CommitParams &p, cudaStream_t stream);

// Chunked tensor-core extend (tcgen05 + TMA), one CTA per (request, head, segment).
// A request's geometry for the persistent extend kernel; the heads of the request share it.
struct alignas(16) ItemRec {
    int b, t0, n, slot;             // request, first token, length, pool slot
    int sp, tslot, nchunks, flags;  // tracked token (n + 1: none) and its slot; chunks; kRec*
};
constexpr int kRecValid = 1;   // a request without faults (the others are skipped)
constexpr int kRecPrefix = 2;  // starts from its pool slot (else from zero)

struct ExtendParams {
    const __nv_bfloat16 *q, *k, *v;
    const float *slopes;
    float *pool;
    const int32_t *state_idx;
    const int32_t *cu_seqlens;
    const uint8_t *prefix_mask;
    __nv_bfloat16 *out;
    unsigned int *err;
    int B, T, H, num_slots, max_seqlen;
    // Grouped-query heads: q and out have H heads; k, v, slopes, the pool and the workspace have
    // Hkv = H / group heads, and query head h reads kv head h / group (group 1: plain).  With
    // group > 1 every query head's CTA carries its kv head's state; the first query head of the
    // group writes the final state, and all of them start from the workspace copy of the
    // initial state (written by the block-state kernel), so that write races no read.
    int Hkv, group;
    unsigned long long wait_limit_ns;  // bound on every mbarrier wait
    // Sequence split of long requests (seg_len == 0: none).  A request of n tokens is cut into
    // segments of seg_len tokens, processed by separate CTAs; segment g starts from
    // e^{-s g seg_len} S0 + sum over the blocks k before it of e^{-s (g seg_len - (k+1) blk_len)} B_k,
    // where B_k is block k's local end state (blk_len tokens, from zero) and S0 the initial state,
    // both written to the workspace by the block-state kernel beforehand; the state scan then
    // leaves that start state in block state g P - 1 (P = seg_len / blk_len).
    int seg_len;   // multiple of blk_len
    int blk_len;   // multiple of the chunk length
    int nseg;      // segments per request, upper bound over the batch
    int nblk;      // blocks per request kept in the workspace
    float *ws;     // [B][Hkv][1 + nblk][D][D]: S0 copy, then block states (segment start states
                   // at every P-th after the scan)
    int lpt;       // nonzero: CTAs take requests longest first (ranked on the device)
    // With lpt: the requests in decreasing length order (ties by index), written by the ranking
    // pre-pass into the workspace for large batches; null: every CTA ranks the (few) requests
    // itself.
    const int32_t *order;
    // Column split (0: none; only without a sequence split).  The csplit longest requests run as
    // two CTAs per head, one per 64-column half of the values, which shortens their chunk chains
    // when the batch leaves SMs idle; the grid has (B + csplit) H CTAs.
    int csplit;
    // Persistent extend: the requests' geometry in decreasing length order (null otherwise).
    const ItemRec *recs;
    // State tracking (both null: none).  For b with track_lens[b] >= 0 the state after the first
    // track_lens[b] tokens of the request is also written to slot track_idx[b]; the CTA that
    // holds that token restarts its chunk grid there and stores the state at that boundary.
    const int32_t *track_lens;
    const int32_t *track_idx;
    // Output layout: element (t, h, j) of out is at t * out_rs + h * out_hs + j (elements); the
    // packed [T][H*D] layout is out_rs = H*D, out_hs = D.
    long long out_rs, out_hs;
};

// Split plan for a batch, from its shape and the device's SM count (seg_len == 0: no split).
struct SplitPlan {
    int seg_len, blk_len, nseg, nblk;
    unsigned long long ws_bytes;
};
// ctas_per_head: CTAs the extend kernel runs per (request, head, segment).
SplitPlan plan_split(int B, int H, int max_seqlen, int num_sms, int ctas_per_head);

cudaError_t launch_extend_wide(const ExtendParams &p, cudaStream_t stream);  // 1 CTA per head

// [T][H*128] bf16 TMA map, box of 64 columns x 128 rows, 128-byte swizzle; rows past T read as
// zero (la_extend_w.cu).
bool make_token_map_full(CUtensorMap *m, const void *ptr, int T, int H);
// The pre-pass of a split or grouped extend: the workspace copy of each initial state, and the
// block states of split requests (la_extend_seg.cu).  Launched when p.seg_len > 0 or p.group > 1.
cudaError_t launch_block_states(const ExtendParams &p, cudaStream_t stream);
// The scan between the two: each split request's block states become, in place, the start states
// of its segments (block g P - 1 holds segment g's), so that the extend kernel reads one matrix per
// segment.  Launched after launch_block_states whenever p.seg_len > 0.
cudaError_t launch_state_scan(const ExtendParams &p, cudaStream_t stream);
// Longest-first order of a batch's requests: order[rank] = request, ranks by decreasing length,
// ties by index (la_extend_seg.cu).  One thread per request compares it with every other.
cudaError_t launch_rank_requests(const int32_t *cu_seqlens, int B, int32_t *order,
                                 cudaStream_t stream);
// Batches above this size keep index order (the ranking's work grows as B^2).
constexpr int kMaxRankedRequests = 65536;

// Persistent extend for batches of more than one wave (la_extend_many.cu): a pre-pass writes one
// ItemRec per request into recs (B of them, in decreasing length order, reporting each faulty
// request once), then `ctas` CTAs work through the (request, head) pairs.  Only for p.group == 1
// without a sequence or column split.
cudaError_t launch_extend_many(const ExtendParams &p, ItemRec *recs, int ctas,
                               cudaStream_t stream);

}  // namespace la
