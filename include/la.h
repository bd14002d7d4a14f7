/*
 * la.h -- C ABI of the GB300 (sm_103a) seg_la library: Bailing-style segmented lightning
 * attention, i.e. per-head linear attention with an ALiBi-style exponential decay.
 *
 * Method source: page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析"
 * (SGLang Lightning Attention capability matrix and seg_la test-coverage analysis), cited as
 * [LA-page].  Its section "独立参考实现：逐 token 递推公式" defines, per head h,
 *     S_t = S_{t-1} * exp(-slope_h) + outer(k_t, v_t)          (S is head_dim x head_dim)
 *     o_t = (q_t @ S_t) * head_dim^-0.5
 * run over each request's tokens, starting from the request's state in a state pool and writing
 * the final state back.
 *
 * Conventions shared by every call
 *   - Element types: q, k, v and out are bfloat16 (passed as their 16-bit patterns, la_bf16);
 *     states and slopes are IEEE fp32; indices are int32; flags are uint8.
 *   - Token layout: a token's row is [H * D] with head h at columns [h*D, (h+1)*D), rows packed
 *     back to back (row stride H*D elements).  This flat [T, H*D] layout is the one the page's
 *     section "生产环境不支持" item 4 describes for the backend's extend and decode output.
 *   - State layout: state_pool is [num_slots][H][D][D] fp32, row-major; in each D x D block the
 *     row index runs over the k dimension and the column index over the v dimension, so
 *     outer(k, v)[i][j] = k_i v_j and (q @ S)[j] = sum_i q_i S[i][j].
 *   - Only head_dim D = 128 is supported (LA_ERR_UNSUPPORTED otherwise), in the spirit of the
 *     head-dim entry guards the page's section "输入与配置覆盖" describes.  q, k and v share one
 *     head count H (no grouped-query heads), as the same section states for seg_la; the _gqa
 *     entry points are the one widening of that, with their own head counts.
 *   - Device pointers to q, k, v, out, state_pool and inter_states must be 16-byte aligned (the
 *     kernels move them with TMA and 16-byte vector accesses), and the fp32 and int32 arrays
 *     (slopes, state_idx, cu_seqlens, parents, accept_idx, track arrays) 4-byte aligned; a call
 *     given a misaligned pointer returns LA_ERR_INVALID before anything is launched.
 *   - Pointers marked "device" must be device memory of the current CUDA device (or managed
 *     memory); "host" pointers are host memory.  The caller owns every buffer; the library keeps
 *     no pointer after a call returns and allocates no device memory.
 *   - Every device call is asynchronous on `stream` (a cudaStream_t; NULL means the legacy
 *     default stream) and does no host synchronisation, so it can be captured in a CUDA graph.
 *     A status of LA_OK means the arguments passed the host checks and the launch succeeded.
 *     Faults the host cannot see (a slot index out of range, inconsistent cu_seqlens, a device
 *     wait that ran out) are recorded in a per-device error word and reported by la_poll_error.
 *   - Preconditions the host cannot check: the state_idx entries of one call are distinct and lie
 *     in [0, num_slots); cu_seqlens is non-decreasing, starts at 0 and ends at T; no request is
 *     longer than max_seqlen; out overlaps no input; inputs are finite.  Out-of-range slots,
 *     inconsistent cu_seqlens and requests longer than max_seqlen are detected on the device
 *     (the affected request is skipped -- nothing of it is written -- and the error word set);
 *     duplicate slots and overlapping buffers give undefined results.
 *   - Argument errors (NULL pointers with B > 0, negative sizes, H < 1, num_slots < 1 ...) return
 *     LA_ERR_INVALID before anything is launched.  B = 0 is a no-op returning LA_OK.
 */
#ifndef LA_GB300_H
#define LA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID = 1,      /* bad argument, detected on the host before any launch */
    LA_ERR_UNSUPPORTED = 2,  /* valid but unsupported configuration (head_dim != 128, ...) */
    LA_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    LA_ERR_TIMEOUT = 4,      /* a bounded device wait ran out (reported by la_poll_error) */
    LA_ERR_DEVICE_INPUT = 5  /* the device found an index out of range: a slot, cu_seqlens, a
                                request longer than max_seqlen, a tree parent, an accept or a
                                track entry (reported by la_poll_error) */
} la_status;

typedef uint16_t la_bf16; /* bfloat16 bit pattern */
typedef void *la_stream;  /* cudaStream_t */

/*
 * la_slopes -- per-head decay slopes for one layer (host only, no device work).
 * [LA-page §独立参考实现], slope bullet: the ALiBi-style slopes times (1 - layer_id/(L-1) + 1e-5),
 * or times (1 + 1e-5) when L = 1.  The ALiBi base is the geometric sequence 2^(-8 (i+1) / H),
 * i = 0..H-1 (the page says only "ALiBi style"; this is that sequence for any H).
 * Computed in double precision and rounded once to fp32.
 *   H         number of heads, >= 1
 *   layer_id  0 <= layer_id < L
 *   L         number of layers, >= 1
 *   host_out  host buffer of H floats, written on success
 * Returns LA_ERR_INVALID for H < 1, L < 1, layer_id outside [0, L) or host_out == NULL.
 */
la_status la_slopes(int H, int layer_id, int L, float *host_out);

/*
 * la_extend -- packed varlen extend (prefill) over the state pool.
 * [LA-page §独立参考实现]: for each request b and head h, start from
 *     S = prefix_mask[b] ? state_pool[state_idx[b], h] : 0
 * run the recurrence over the request's tokens, write o_t to out, and write the final S back to
 * state_pool[state_idx[b], h] (also when prefix_mask[b] = 0, and for zero-length requests).
 *   q, k, v      device, bf16 [T][H*D]; request b owns rows [cu_seqlens[b], cu_seqlens[b+1])
 *   slopes       device, fp32 [H] (for example from la_slopes)
 *   state_pool   device, fp32 [num_slots][H][D][D], read and updated in place; only the slots
 *                named in state_idx are touched
 *   num_slots    number of pool slots, >= 1
 *   state_idx    device, int32 [B]
 *   cu_seqlens   device, int32 [B+1]
 *   prefix_mask  device, uint8 [B]; nonzero = start from the pool slot, 0 = start from zero
 *                (the slot is then never read)
 *   out          device, bf16 [T][H*D], written
 *   B, T, H, D   requests, total tokens (= cu_seqlens[B]), heads, head_dim (must be 128)
 *   max_seqlen   an upper bound on every request's length (T is always a valid value); it and
 *                B, H decide the schedule (see la_extend_workspace_size).  A request longer than
 *                max_seqlen is skipped (no output rows, no state written) and la_poll_error
 *                reports LA_ERR_DEVICE_INPUT.
 *   workspace    device scratch of workspace_bytes bytes (16-byte aligned), or NULL.  (This
 *                argument pair extends the plain call with a caller-owned scratch buffer, so
 *                that the library itself never allocates.)  When the
 *                batch has too few (request, head) pairs to fill the GPU, long requests are cut
 *                into segments processed in parallel; that needs la_extend_workspace_size()
 *                bytes of scratch.  With NULL or a smaller buffer the call runs without that
 *                split (same results up to rounding, fewer CTAs).  The caller owns it; its
 *                contents on entry do not matter and are garbage on exit; calls sharing one
 *                workspace must not overlap on the GPU.  Without the sequence split, SMs left
 *                idle may take the longest requests as two CTAs per head (la_set_column_split);
 *                that needs no scratch.  A batch of more (request, head) pairs than SMs runs on
 *                a persistent grid of one CTA per SM (la_set_persistent), which keeps B records
 *                of 32 bytes in the workspace; without them it runs one CTA per pair, in waves
 *                (same results, bit for bit).  A batch of 2 .. 256 requests whose B * H pairs fit
 *                on the SMs, that has no sequence split and whose max_seqlen is at least twice
 *                its mean length T / B, runs balanced when the workspace has room for its plan
 *                (la_set_balanced): a one-block planner on the device cuts the
 *                longest requests into segments from their actual lengths, each segment's CTA
 *                first forms its start state from the request's earlier keys and values, and a
 *                persistent grid of one CTA per SM works through the segments (about 13 KiB of
 *                plan in the workspace; same results up to rounding).
 *   workspace_bytes  size of workspace
 *   stream       cudaStream_t
 * Numerics: bf16 inputs; fp32 states and accumulation.  Every product runs on the tensor cores
 * in bf16 with fp32 accumulation, and the three operands the kernel computes -- the decay-masked
 * scores P, the decayed keys lambda K and the state for Q S -- each as a bf16 pair hi + lo (about
 * 2^-17 together); out is rounded to bf16 once.
 */
la_status la_extend(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                    float *state_pool, int num_slots, const int32_t *state_idx,
                    const int32_t *cu_seqlens, const uint8_t *prefix_mask, la_bf16 *out, int B,
                    int T, int H, int D, int max_seqlen, void *workspace, size_t workspace_bytes,
                    la_stream stream);

/*
 * la_extend_ex -- la_extend with two options: a state-tracking snapshot per request, and the
 * layout of out.
 *
 * State tracking ([LA-page §额外覆盖], the extra-buffer state tracking of a prefill: at the
 * track_len-th token the running state is copied into a track slot, while the request's own slot
 * still receives the final state and no other slot is written):
 *   track_lens       device, int32 [B]: the snapshot is the state after the first track_lens[b]
 *                    tokens of request b in this call (0: its initial state -- the prefix state
 *                    or zero; its length: its final state); -1: no snapshot for b
 *   track_state_idx  device, int32 [B]: the pool slot that receives b's snapshot (ignored when
 *                    track_lens[b] == -1)
 * Both NULL: no snapshots.  One NULL: LA_ERR_INVALID.  A track length outside [-1, length] or a
 * track slot that is out of range or equal to the request's own slot skips that snapshot and is
 * reported by la_poll_error as LA_ERR_DEVICE_INPUT.  Track slots must differ from every slot the
 * call reads or writes otherwise and from one another (not checked: overlapping slots race).  The
 * request's chunk grid is restarted at the tracked token, so the snapshot is the state the
 * kernel carries at that chunk boundary (one more, partial, chunk); outputs and final states
 * equal la_extend's up to rounding, bit for bit for a request whose track length is -1, its
 * length, or a multiple of 128.
 *
 * Output layout ([LA-page §生产环境不支持, item 4]: the backend returns out flattened to
 * [T, H*D] while the piecewise-CUDA-graph path writes a per-head [T, H, D] buffer; this lets out
 * be any such buffer, including a strided view):
 *   out_row_stride   elements from token t to token t+1 in out (0: H*D, the packed layout)
 *   out_head_stride  elements from head h to head h+1 in out (0: D)
 * Element j of head h of token t goes to out[t * out_row_stride + h * out_head_stride + j].  Both
 * strides must be multiples of 8 (16-byte aligned stores), and rows of heads or heads of rows must
 * not overlap (out_row_stride >= (H-1) * out_head_stride + D, or out_head_stride >=
 * (T-1) * out_row_stride + D); LA_ERR_INVALID otherwise.  Elements between the written ones are
 * left untouched.  A contiguous [T, H, D] buffer is the packed layout.
 *
 * All other arguments, the launches and the errors are those of la_extend.  With no snapshots and
 * the packed layout this is la_extend.
 */
la_status la_extend_ex(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                       float *state_pool, int num_slots, const int32_t *state_idx,
                       const int32_t *cu_seqlens, const uint8_t *prefix_mask,
                       const int32_t *track_lens, const int32_t *track_state_idx, la_bf16 *out,
                       int64_t out_row_stride, int64_t out_head_stride, int B, int T, int H, int D,
                       int max_seqlen, void *workspace, size_t workspace_bytes, la_stream stream);

/*
 * la_extend_workspace_size -- bytes of device scratch la_extend would use for a batch of this
 * shape on the current device: the block states of a sequence split, the longest-first order of a
 * batch of more than 256 requests, the request records of the persistent grid (0 when it needs
 * none of these).  Host only, no device work
 * beyond one cached attribute query.  Arguments as for la_extend; *bytes is written on success.
 * Returns LA_ERR_INVALID for negative sizes or bytes == NULL, LA_ERR_UNSUPPORTED for D != 128.
 */
la_status la_extend_workspace_size(int B, int T, int H, int D, int max_seqlen, size_t *bytes);

/*
 * la_extend_noalloc -- la_extend for callers that cannot allocate device memory.
 * No counterpart on the paper: this is a convenience of this library.  la_extend may need scratch
 * memory for long requests in small batches (see la_extend_workspace_size), which the caller must
 * allocate; a caller that cannot -- a plugin inside a host framework that owns the device's memory
 * budget and hands over only input and output buffers, or a latency-critical loop that must not
 * call cudaMalloc -- uses this entry point instead.  It takes la_extend's arguments without the
 * workspace and computes the same result, using a fixed 16 MiB scratch array that the library
 * keeps in device memory on every device that loads it (held until the process exits).
 *   - It allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *   - A batch whose split plan needs more than 16 MiB of scratch is rejected with
 *     LA_ERR_UNSUPPORTED before anything is launched.  The largest plan is 1.5 x (SM count)
 *     matrices of 64 KiB -- 14.25 MiB on a 152-SM GB300 -- so every plan fits on devices of up to
 *     170 SMs; use la_extend with a workspace otherwise.  (The balanced schedule's plan, for
 *     skewed one-wave batches, takes about 13 KiB.)
 *   - The first call on a device looks up the array's device address and caches it; make that
 *     first call before any stream capture.  Do not use it again in a process after
 *     cudaDeviceReset (the cached address belongs to the old context).
 *   - All calls on a device share the array and it keeps the last call's contents; nothing in it
 *     needs to start at zero, but calls that overlap on the GPU race on it: serialise them.
 */
la_status la_extend_noalloc(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v,
                            const float *slopes, float *state_pool, int num_slots,
                            const int32_t *state_idx, const int32_t *cu_seqlens,
                            const uint8_t *prefix_mask, la_bf16 *out, int B, int T, int H, int D,
                            int max_seqlen, la_stream stream);

/*
 * la_extend_gqa -- la_extend with grouped-query heads: H query heads share Hkv key/value heads.
 * The page's section "输入与配置覆盖" notes that seg_la takes one head count for q, k and v (no
 * grouped-query attention); this entry point is that widening, and la_extend stays the page's
 * plain form.  The state is a property of the key/value stream, so there is one state and one
 * slope per kv head: for request b and kv head j, S^(j) follows the recurrence of
 * [LA-page §独立参考实现] with k^(j), v^(j) and slopes[j], and query head h of the group
 * j = h / (H / Hkv) reads it out, o_t^(h) = (q_t^(h) @ S_t^(j)) * D^-0.5.  With Hkv = H this is
 * la_extend, bit for bit.
 *   q, out       device, bf16 [T][H*D]
 *   k, v         device, bf16 [T][Hkv*D]
 *   slopes       device, fp32 [Hkv]
 *   state_pool   device, fp32 [num_slots][Hkv][D][D]
 *   H, Hkv       query heads and kv heads; H must be a multiple of Hkv (LA_ERR_INVALID otherwise)
 *   workspace    device scratch of at least la_extend_gqa_workspace_size() bytes when Hkv < H
 *                (each kv head's initial state is copied there first, so that the group's first
 *                query head can write the final state back while the others still start from
 *                the copy); LA_ERR_INVALID when it is missing or smaller than the copies need.
 *                The rest of the scratch, when present, lets long requests be split as in
 *                la_extend.
 * All other arguments, the checks and the errors are those of la_extend.  Each query head's CTA
 * carries its kv head's state, so the kv-side work is repeated per query head; the K and V tiles
 * the group's CTAs read at about the same time come from L2.
 */
la_status la_extend_gqa(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                        float *state_pool, int num_slots, const int32_t *state_idx,
                        const int32_t *cu_seqlens, const uint8_t *prefix_mask, la_bf16 *out,
                        int B, int T, int H, int Hkv, int D, int max_seqlen, void *workspace,
                        size_t workspace_bytes, la_stream stream);

/*
 * la_extend_gqa_workspace_size -- bytes of device scratch la_extend_gqa uses for a batch of this
 * shape on the current device: the initial-state copies (B * Hkv matrices of D x D fp32) when
 * Hkv < H, plus the split plan's block states when long requests are split; 0 when Hkv = H and
 * nothing is split.  Host only.  LA_ERR_INVALID for bad sizes or bytes == NULL.
 */
la_status la_extend_gqa_workspace_size(int B, int T, int H, int Hkv, int D, int max_seqlen,
                                       size_t *bytes);

/*
 * la_decode_gqa -- la_decode with grouped-query heads (see la_extend_gqa): one decode token per
 * request; kv head j's state is advanced once, in place, and read out by each of its H / Hkv
 * query heads.  One CTA per (request, kv head) does both, so a state crosses HBM once however
 * many query heads share it.  q, out: device bf16 [B][H*D]; k, v: [B][Hkv*D]; slopes [Hkv];
 * state_pool [num_slots][Hkv][D][D].  With Hkv = H this is la_decode.  Checks and errors as for
 * la_decode; H must be a multiple of Hkv.
 */
la_status la_decode_gqa(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                        float *state_pool, int num_slots, const int32_t *state_idx, la_bf16 *out,
                        int B, int H, int Hkv, int D, la_stream stream);

/*
 * la_decode -- one decode token per request, state updated in place.
 * The recurrence of [LA-page §独立参考实现] for a single token; the page's section
 * "输入与配置覆盖" names the matching decode kernel.  For each request b and head h:
 *     S = state_pool[state_idx[b], h];  S = S * exp(-slopes[h]) + outer(k_b, v_b);
 *     out_b = (q_b @ S) * D^-0.5;       state_pool[state_idx[b], h] = S
 *   q, k, v     device, bf16 [B][H*D]
 *   slopes      device, fp32 [H]
 *   state_pool  device, fp32 [num_slots][H][D][D], updated in place (named slots only)
 *   state_idx   device, int32 [B]
 *   out         device, bf16 [B][H*D], written
 */
la_status la_decode(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v, const float *slopes,
                    float *state_pool, int num_slots, const int32_t *state_idx, la_bf16 *out,
                    int B, int H, int D, la_stream stream);

/*
 * la_verify_chain -- chain (topk = 1) target verify of N draft tokens per request.
 * [LA-page §生产环境不支持, item 3]: seg_la treats draft tokens as a chain, each one continuing
 * from the previous position's state (the page's backend refuses topk > 1; la_verify_tree below
 * is this library's tree variant).  For each request b and head h, from
 * S = state_pool[state_idx[b], h], for t = 0..N-1: apply the recurrence to token b*N + t, write
 * its output row, and store S into inter_states[b][t][h].  The pool is only read; committing an
 * accepted draft state is the caller's copy from inter_states.
 *   q, k, v       device, bf16 [B*N][H*D] (request-major: request b owns rows b*N .. b*N+N-1)
 *   slopes        device, fp32 [H]
 *   state_pool    device, fp32 [num_slots][H][D][D], read only
 *   state_idx     device, int32 [B]
 *   inter_states  device, fp32 [B][N][H][D][D], written
 *   out           device, bf16 [B*N][H*D], written
 *   N             draft tokens per request, >= 1
 */
la_status la_verify_chain(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v,
                          const float *slopes, const float *state_pool, int num_slots,
                          const int32_t *state_idx, float *inter_states, la_bf16 *out, int B,
                          int N, int H, int D, la_stream stream);

/*
 * la_verify_tree -- tree target verify (EAGLE-style, topk > 1) of N draft tokens per request.
 * [LA-page §生产环境不支持, item 3 and §Next Work, item 2]: the page's seg_la handles draft tokens
 * only as a chain and names the kernel-level fix -- each draft token forks from the state saved
 * for its parent.  This call is that fix: for each request b and head h, draft token t continues
 * from the state after token parents[b*N + t] (from state_pool[state_idx[b], h] when that is -1),
 * its output row is written and its state stored into inter_states[b][t][h].  A chain
 * (parents[t] = t - 1) gives exactly la_verify_chain's results.  The pool is only read.
 *   parents       device, int32 [B][N]; each entry in [-1, t-1] (topologically ordered tree)
 *   other arguments as for la_verify_chain
 * A request with a parent outside [-1, t-1] is skipped (nothing written) and la_poll_error
 * reports LA_ERR_DEVICE_INPUT.
 */
la_status la_verify_tree(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v,
                         const float *slopes, const float *state_pool, int num_slots,
                         const int32_t *state_idx, const int32_t *parents, float *inter_states,
                         la_bf16 *out, int B, int N, int H, int D, la_stream stream);

/*
 * la_commit_accepted -- after a verify call, move the state of the last accepted draft token of
 * each request into its pool slot: state_pool[state_idx[b], h] = inter_states[b][accept_idx[b]][h]
 * for every head, when accept_idx[b] >= 0 (-1: nothing accepted, the slot is left as is).  With
 * chain verify accept_idx[b] is (number of accepted tokens - 1); with tree verify it is the last
 * node of the accepted path.  The verify calls leave the pool alone ([LA-page §生产环境不支持,
 * item 3]: the page's intermediate-state pipeline is per request); this is the commit step that
 * completes them.
 *   inter_states  device, fp32 [B][N][H][D][D] (as written by la_verify_chain / la_verify_tree)
 *   accept_idx    device, int32 [B], each in [-1, N-1]
 *   state_pool    device, fp32 [num_slots][H][D][D], updated in place (named slots only)
 *   state_idx     device, int32 [B]
 * An index outside [-1, N-1] or a slot out of range skips that request and is reported by
 * la_poll_error as LA_ERR_DEVICE_INPUT.
 */
la_status la_commit_accepted(const float *inter_states, const int32_t *accept_idx,
                             float *state_pool, int num_slots, const int32_t *state_idx, int B,
                             int N, int H, int D, la_stream stream);

/*
 * la_poll_error -- synchronise `stream` and then the whole current device (every stream on it),
 * then read and clear the device's error word.  The word is shared by all of the library's
 * kernels on the device, whatever stream they run on, so the device-wide synchronisation makes
 * sure that a fault recorded by a kernel still running on another stream is neither missed nor
 * reported by a later poll.  Returns LA_ERR_TIMEOUT if a bounded device wait ran out,
 * LA_ERR_DEVICE_INPUT if a kernel found a slot index out of range, inconsistent cu_seqlens, a
 * request longer than max_seqlen, a tree parent, commit index or track entry out of range,
 * LA_ERR_CUDA if a CUDA error is pending, else LA_OK.  This is the one call that blocks the host
 * (and it cannot be captured in a CUDA graph).
 */
la_status la_poll_error(la_stream stream);

/* la_status_string -- static, human-readable name of a status code (never NULL). */
const char *la_status_string(la_status status);

/*
 * la_set_wait_limit -- diagnostics: how long (in microseconds) a device wait inside the extend
 * kernel may last before it gives up, sets the error word (LA_ERR_TIMEOUT from la_poll_error)
 * and lets the kernel exit cleanly: the CTA waits for its own copies and MMAs in flight, frees
 * its tensor memory and returns, leaving the context usable.  0 restores the default (2 s, far
 * above any legitimate wait).  Host only; applies to later launches from this process.  Lets a
 * test drive the timeout path without hanging or faulting the GPU.
 */
void la_set_wait_limit(uint64_t microseconds);

/*
 * la_set_column_split -- scheduling switch for la_extend / la_extend_ex (default 1: on).  When a
 * call runs without a sequence split and its B * H CTAs leave at least H of the device's SMs
 * idle, the longest requests (as many as the idle SMs allow, H CTAs each) run as two CTAs per
 * head, each on one 64-column half of the values, which shortens the longest chunk chains.  The
 * result is the same up to rounding either way.  0 runs one CTA per (request, head) always.
 * Host only; applies to later launches from this process.
 */
void la_set_column_split(int enable);

/*
 * la_set_persistent -- scheduling switch for la_extend / la_extend_ex (default 1: on).  A batch
 * whose B * H (request, head) pairs outnumber the device's SMs runs, when the workspace has room
 * for its request records, on a persistent grid: one CTA per SM works through its share of the
 * pairs (longest first, dealt in snake order), keeping its barriers and tensor memory and loading
 * the next pair's tiles while it finishes the current one.  Every pair is computed as one CTA per
 * pair computes it, so the results are bit-identical either way.  0 runs one CTA per pair always.
 * Grouped-query calls always run one CTA per pair.  Host only; applies to later launches from
 * this process.
 */
void la_set_persistent(int enable);

/*
 * la_set_balanced -- scheduling switch for la_extend / la_extend_ex (default 1: on).  A batch of
 * 2 .. 256 requests whose B * H (request, head) pairs fit on the device's SMs, that has no
 * sequence split and whose max_seqlen is at least twice its mean length T / B (a few long
 * requests among short ones), runs, when the workspace has room for the plan, as segments planned on the
 * device: the longest requests are cut so that every SM gets about the same number of chunks
 * (each segment's CTA first forms the state at its start from the request's earlier keys and
 * values, reading them a second time), and one CTA per SM works through the segments.  The
 * result is the same up to rounding either way (the start state of a segment sums the same terms
 * in another grouping).  0 keeps one CTA per (request, head), with the column split.  Grouped-
 * query calls never run balanced.  Host only; applies to later launches from this process.
 */
void la_set_balanced(int enable);

#ifdef __cplusplus
}
#endif

#endif /* LA_GB300_H */
