/*
 * la_oracle.c -- fp64 CPU oracle for Bailing-style segmented lightning attention (seg_la).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this file: only the
 * tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares no code, header or
 * table with the CUDA library; both sides see only the same seeded inputs.
 *
 * Source of the method.  Page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析"
 * (SGLang Lightning Attention capability matrix and seg_la test-coverage analysis), cited below as
 * [LA-page].  Sections used:
 *   [LA-page §独立参考实现]  "Independent reference implementation: per-token recurrence formula":
 *       per head h:  state_t = state_{t-1} * exp(-slope_h) + outer(k_t, v_t)
 *                    o_t     = q_t @ state_t * head_dim ** -0.5
 *       looped token by token per request, final state written back at the end; prefix requests
 *       start from a state injected into the state pool; the slope rule
 *       slopes * (1 - layer_id/(L-1) + 1e-5), and slopes * (1 + 1e-5) when L = 1.
 *   [LA-page §生产环境不支持 item 3]  chain (topk = 1) target verify: every draft token continues
 *       from the previous position's state; once the target model has accepted some draft
 *       tokens, the state after the last accepted one becomes the request's state.
 *   [LA-page §额外覆盖]  "extra coverage: state tracking": during a prefill, the state at the
 *       track_len-th token is also copied into a separate track slot, while the request's own
 *       slot still receives the final state and every other slot is left alone.
 *   [LA-page §Next Work, item 2]  tree verify: each draft token forks from the state saved for
 *       its parent, not from the previous position of the chain.
 *
 * Everything is evaluated in double precision straight from those definitions: no chunking, no
 * blocking, no reassociation.  The state is S[i][j] with i on the k index (rows) and j on the v
 * index (columns), so outer(k, v)[i][j] = k_i * v_j and (q @ S)[j] = sum_i q_i * S[i][j].
 *
 * Readings of points the page leaves open (each also listed in the design notes):
 *   - base slopes are the ALiBi geometric sequence 2^(-8 (i+1) / H), i = 0..H-1;
 *   - decay is applied before the outer product is added, so the current token has weight 1;
 *   - a request whose prefix flag is 0 starts from the zero state and never reads its slot;
 *   - the final state is written back for every request, including zero-length ones;
 *   - state tracking: "the state at the track_len-th token" is the state after the first
 *     track_len tokens of this call (track_len counts the call's new tokens, 0 meaning the
 *     initial state); -1 means no snapshot; the track slot is a slot of the same pool and must
 *     not be the request's own slot;
 *   - chain verify leaves the pool untouched and records the state after each draft token;
 *   - tree verify: parent[t] in [-1, t-1], -1 meaning the request's pool state; the state after
 *     token t is the recurrence applied to token t from the state after its parent;
 *   - grouped-query heads (a widening the page's section "输入与配置覆盖" says seg_la lacks: it
 *     takes one head count for q, k and v): with H query heads and Hkv key/value heads (H a
 *     multiple of Hkv, G = H / Hkv), query head h belongs to kv head j = h / G.  The state is a
 *     property of the key/value stream, so there is one state and one slope per kv head: S^(j)
 *     follows the page's recurrence with k^(j), v^(j) and slope_j, and every query head of the
 *     group reads the same S^(j) out.  With Hkv = H this is the plain recurrence.
 *
 * Threads: the (request, head) pairs are independent, so they are spread over POSIX threads.
 * This changes no arithmetic: every pair is still one plain sequential loop.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* [LA-page §独立参考实现], the slope bullet: ALiBi-style per-head slope times the per-layer factor. */
void la_oracle_slopes(int H, int layer_id, int L, double *out)
{
    double factor;
    if (L == 1)
        factor = 1.0 + 1e-5;
    else
        factor = 1.0 - (double)layer_id / (double)(L - 1) + 1e-5;
    for (int i = 0; i < H; i++)
        out[i] = pow(2.0, -8.0 * (double)(i + 1) / (double)H) * factor;
}

/* One request-head recurrence over n tokens, starting from S (in place).
 * q, k, v point at the first token's head slice; row_stride is the distance between tokens.
 * If inter != NULL, the state after token t is copied to inter + t * inter_stride. */
static void recur(double *S, int D, double slope, int n, const double *q, const double *k,
                  const double *v, size_t row_stride, double *out, double *inter,
                  size_t inter_stride)
{
    const double decay = exp(-slope);
    const double scale = 1.0 / sqrt((double)D);
    for (int t = 0; t < n; t++) {
        const double *qt = q + (size_t)t * row_stride;
        const double *kt = k + (size_t)t * row_stride;
        const double *vt = v + (size_t)t * row_stride;
        /* state_t = state_{t-1} * exp(-slope) + outer(k_t, v_t) */
        for (int i = 0; i < D; i++)
            for (int j = 0; j < D; j++)
                S[(size_t)i * D + j] = S[(size_t)i * D + j] * decay + kt[i] * vt[j];
        /* o_t = q_t @ state_t * head_dim^-0.5 */
        double *ot = out + (size_t)t * row_stride;
        for (int j = 0; j < D; j++) {
            double acc = 0.0;
            for (int i = 0; i < D; i++)
                acc += qt[i] * S[(size_t)i * D + j];
            ot[j] = acc * scale;
        }
        if (inter)
            memcpy(inter + (size_t)t * inter_stride, S, sizeof(double) * (size_t)D * D);
    }
}

enum { OP_EXTEND = 0, OP_DECODE = 1, OP_VERIFY = 2 };

typedef struct {
    int op;
    const double *q, *k, *v, *slopes;
    double *pool;                 /* [num_slots][H][D][D] */
    const int32_t *state_idx;     /* [B] */
    const int32_t *cu_seqlens;    /* [B+1] (extend) */
    const uint8_t *prefix_mask;   /* [B]   (extend) */
    double *out;                  /* [T][H*D] */
    double *inter;                /* [B][N][H][D][D] (verify) */
    const int32_t *track_lens;    /* [B] or NULL (extend with state tracking) */
    const int32_t *track_idx;     /* [B] or NULL */
    int B, H, D, N;
    int nthreads;
    int tid;
} job_t;

static void run_pair(const job_t *a, int b, int h)
{
    const int D = a->D, H = a->H;
    const size_t row = (size_t)H * D, dd = (size_t)D * D;
    double *slot = a->pool + ((size_t)a->state_idx[b] * H + h) * dd;
    double *S = (double *)malloc(sizeof(double) * dd);
    if (a->op == OP_EXTEND) {
        /* [LA-page §独立参考实现], prefix-state injection: prefix requests start from the pool. */
        if (a->prefix_mask[b])
            memcpy(S, slot, sizeof(double) * dd);
        else
            memset(S, 0, sizeof(double) * dd);
        const int t0 = a->cu_seqlens[b], n = a->cu_seqlens[b + 1] - t0;
        const size_t off = (size_t)t0 * row + (size_t)h * D;
        /* [LA-page §额外覆盖] state tracking: once the first track_len tokens are processed,
         * the state of that moment is copied into the track slot; the run then goes on. */
        const int tl = a->track_lens ? a->track_lens[b] : -1;
        const int n1 = tl >= 0 ? tl : n;
        recur(S, D, a->slopes[h], n1, a->q + off, a->k + off, a->v + off, row, a->out + off,
              NULL, 0);
        if (tl >= 0) {
            memcpy(a->pool + ((size_t)a->track_idx[b] * H + h) * dd, S, sizeof(double) * dd);
            const size_t off2 = off + (size_t)n1 * row;
            recur(S, D, a->slopes[h], n - n1, a->q + off2, a->k + off2, a->v + off2, row,
                  a->out + off2, NULL, 0);
        }
        memcpy(slot, S, sizeof(double) * dd); /* final state written back at the end */
    } else if (a->op == OP_DECODE) {
        memcpy(S, slot, sizeof(double) * dd);
        const size_t off = (size_t)b * row + (size_t)h * D;
        recur(S, D, a->slopes[h], 1, a->q + off, a->k + off, a->v + off, row, a->out + off,
              NULL, 0);
        memcpy(slot, S, sizeof(double) * dd);
    } else {
        /* chain verify: token t of request b continues from token t-1; pool is only read */
        memcpy(S, slot, sizeof(double) * dd);
        const size_t off = (size_t)b * a->N * row + (size_t)h * D;
        double *inter = a->inter + ((size_t)b * a->N * H + h) * dd;
        recur(S, D, a->slopes[h], a->N, a->q + off, a->k + off, a->v + off, row, a->out + off,
              inter, (size_t)H * dd);
    }
    free(S);
}

static void *worker(void *p)
{
    const job_t *a = (const job_t *)p;
    const int pairs = a->B * a->H;
    for (int w = a->tid; w < pairs; w += a->nthreads)
        run_pair(a, w / a->H, w % a->H);
    return NULL;
}

static int run(job_t *a)
{
    int nt = a->nthreads < 1 ? 1 : a->nthreads;
    if (nt > a->B * a->H)
        nt = a->B * a->H > 0 ? a->B * a->H : 1;
    if (nt == 1) {
        a->nthreads = 1;
        a->tid = 0;
        worker(a);
        return 0;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * nt);
    for (int i = 0; i < nt; i++) {
        jobs[i] = *a;
        jobs[i].nthreads = nt;
        jobs[i].tid = i;
        if (pthread_create(&th[i], NULL, worker, &jobs[i]) != 0) {
            /* fall back to running this share on the calling thread */
            worker(&jobs[i]);
            th[i] = 0;
        }
    }
    for (int i = 0; i < nt; i++)
        if (th[i])
            pthread_join(th[i], NULL);
    free(th);
    free(jobs);
    return 0;
}

/* Packed varlen extend: q, k, v, out are [T][H*D]; request b covers rows
 * [cu_seqlens[b], cu_seqlens[b+1]); its state lives in pool[state_idx[b]]. */
int la_oracle_extend(const double *q, const double *k, const double *v, const double *slopes,
                     double *pool, const int32_t *state_idx, const int32_t *cu_seqlens,
                     const uint8_t *prefix_mask, double *out, int B, int H, int D, int nthreads)
{
    job_t a = {0};
    a.op = OP_EXTEND;
    a.q = q; a.k = k; a.v = v; a.slopes = slopes; a.pool = pool;
    a.state_idx = state_idx; a.cu_seqlens = cu_seqlens; a.prefix_mask = prefix_mask;
    a.out = out; a.B = B; a.H = H; a.D = D; a.N = 0; a.nthreads = nthreads;
    return run(&a);
}

/* Extend with state tracking: as la_oracle_extend, and for every request b with
 * track_lens[b] >= 0 the state after its first track_lens[b] tokens (its initial state when 0,
 * its final state when track_lens[b] is its length) is also written to pool slot track_idx[b].
 * track_lens[b] == -1: no snapshot.  Returns -1 (and computes nothing) if some track_lens[b] is
 * outside [-1, length of b] or a snapshot would go to the request's own slot. */
int la_oracle_extend_tracked(const double *q, const double *k, const double *v,
                             const double *slopes, double *pool, const int32_t *state_idx,
                             const int32_t *cu_seqlens, const uint8_t *prefix_mask,
                             const int32_t *track_lens, const int32_t *track_idx, double *out,
                             int B, int H, int D, int nthreads)
{
    for (int b = 0; b < B; b++) {
        const int tl = track_lens[b], n = cu_seqlens[b + 1] - cu_seqlens[b];
        if (tl < -1 || tl > n || (tl >= 0 && track_idx[b] == state_idx[b]))
            return -1;
    }
    job_t a = {0};
    a.op = OP_EXTEND;
    a.q = q; a.k = k; a.v = v; a.slopes = slopes; a.pool = pool;
    a.state_idx = state_idx; a.cu_seqlens = cu_seqlens; a.prefix_mask = prefix_mask;
    a.track_lens = track_lens; a.track_idx = track_idx;
    a.out = out; a.B = B; a.H = H; a.D = D; a.N = 0; a.nthreads = nthreads;
    return run(&a);
}

/* One-token decode: q, k, v, out are [B][H*D]; every request starts from its pool slot and the
 * slot is updated in place. */
int la_oracle_decode(const double *q, const double *k, const double *v, const double *slopes,
                     double *pool, const int32_t *state_idx, double *out, int B, int H, int D,
                     int nthreads)
{
    job_t a = {0};
    a.op = OP_DECODE;
    a.q = q; a.k = k; a.v = v; a.slopes = slopes; a.pool = pool; a.state_idx = state_idx;
    a.out = out; a.B = B; a.H = H; a.D = D; a.nthreads = nthreads;
    return run(&a);
}

/* Tree verify: like chain verify, but draft token t of request b continues from the state after
 * token parents[b*N + t] (or from the pool state when that is -1); parents must point backwards.
 * Returns -1 (and computes nothing) if some parent is out of [-1, t-1]. */
int la_oracle_verify_tree(const double *q, const double *k, const double *v, const double *slopes,
                          const double *pool, const int32_t *state_idx, const int32_t *parents,
                          double *inter, double *out, int B, int N, int H, int D)
{
    for (int b = 0; b < B; b++)
        for (int t = 0; t < N; t++)
            if (parents[(size_t)b * N + t] < -1 || parents[(size_t)b * N + t] >= t)
                return -1;
    const size_t row = (size_t)H * D, dd = (size_t)D * D;
    const double scale = 1.0 / sqrt((double)D);
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            const double decay = exp(-slopes[h]);
            const double *root = pool + ((size_t)state_idx[b] * H + h) * dd;
            for (int t = 0; t < N; t++) {
                const int par = parents[(size_t)b * N + t];
                const double *base =
                    par < 0 ? root : inter + (((size_t)b * N + par) * H + h) * dd;
                double *S = inter + (((size_t)b * N + t) * H + h) * dd;
                const size_t off = ((size_t)b * N + t) * row + (size_t)h * D;
                const double *qt = q + off, *kt = k + off, *vt = v + off;
                for (int i = 0; i < D; i++)
                    for (int j = 0; j < D; j++)
                        S[(size_t)i * D + j] = base[(size_t)i * D + j] * decay + kt[i] * vt[j];
                for (int j = 0; j < D; j++) {
                    double acc = 0.0;
                    for (int i = 0; i < D; i++)
                        acc += qt[i] * S[(size_t)i * D + j];
                    out[off + j] = acc * scale;
                }
            }
        }
    }
    return 0;
}

/* Chain verify: q, k, v, out are [B*N][H*D] (request-major, N draft tokens each); the pool is
 * read only; inter is [B][N][H][D][D], the state after each draft token. */
int la_oracle_verify_chain(const double *q, const double *k, const double *v,
                           const double *slopes, const double *pool, const int32_t *state_idx,
                           double *inter, double *out, int B, int N, int H, int D, int nthreads)
{
    job_t a = {0};
    a.op = OP_VERIFY;
    a.q = q; a.k = k; a.v = v; a.slopes = slopes; a.pool = (double *)pool;
    a.state_idx = state_idx; a.inter = inter; a.out = out;
    a.B = B; a.H = H; a.D = D; a.N = N; a.nthreads = nthreads;
    return run(&a);
}

/* ---------------------------------------------------------------- grouped-query heads
 * One kv head's recurrence over n tokens from S (in place), read out by its G query heads.
 * qg, og point at the group's first query head of the first token (query head g at + g*D);
 * kj, vj at the kv head's slice of the first token.  Per token the state is advanced once and
 * then read out once per query head. */
static void recur_group(double *S, int D, double slope, int n, int G, const double *qg,
                        size_t q_stride, const double *kj, const double *vj, size_t kv_stride,
                        double *og)
{
    const double decay = exp(-slope);
    const double scale = 1.0 / sqrt((double)D);
    for (int t = 0; t < n; t++) {
        const double *kt = kj + (size_t)t * kv_stride;
        const double *vt = vj + (size_t)t * kv_stride;
        /* state_t = state_{t-1} * exp(-slope_j) + outer(k_t, v_t), once per kv head */
        for (int i = 0; i < D; i++)
            for (int j = 0; j < D; j++)
                S[(size_t)i * D + j] = S[(size_t)i * D + j] * decay + kt[i] * vt[j];
        /* o_t^(h) = q_t^(h) @ state_t * head_dim^-0.5 for each query head of the group */
        for (int g = 0; g < G; g++) {
            const double *qt = qg + (size_t)t * q_stride + (size_t)g * D;
            double *ot = og + (size_t)t * q_stride + (size_t)g * D;
            for (int j = 0; j < D; j++) {
                double acc = 0.0;
                for (int i = 0; i < D; i++)
                    acc += qt[i] * S[(size_t)i * D + j];
                ot[j] = acc * scale;
            }
        }
    }
}

typedef struct {
    int decode;
    const double *q, *k, *v, *slopes;
    double *pool;                 /* [num_slots][Hkv][D][D] */
    const int32_t *state_idx, *cu_seqlens;
    const uint8_t *prefix_mask;
    double *out;                  /* [rows][H*D] */
    int B, H, Hkv, D, nthreads, tid;
} gqa_job_t;

static void *gqa_worker(void *p)
{
    const gqa_job_t *a = (const gqa_job_t *)p;
    const int D = a->D, G = a->H / a->Hkv;
    const size_t q_row = (size_t)a->H * D, kv_row = (size_t)a->Hkv * D, dd = (size_t)D * D;
    double *S = (double *)malloc(sizeof(double) * dd);
    for (int w = a->tid; w < a->B * a->Hkv; w += a->nthreads) {
        const int b = w / a->Hkv, j = w % a->Hkv;
        double *slot = a->pool + ((size_t)a->state_idx[b] * a->Hkv + j) * dd;
        int t0, n;
        if (a->decode) {
            t0 = b;
            n = 1;
            memcpy(S, slot, sizeof(double) * dd);
        } else {
            t0 = a->cu_seqlens[b];
            n = a->cu_seqlens[b + 1] - t0;
            if (a->prefix_mask[b])
                memcpy(S, slot, sizeof(double) * dd);
            else
                memset(S, 0, sizeof(double) * dd);
        }
        const size_t qo = (size_t)t0 * q_row + (size_t)j * G * D;
        const size_t kvo = (size_t)t0 * kv_row + (size_t)j * D;
        recur_group(S, D, a->slopes[j], n, G, a->q + qo, q_row, a->k + kvo, a->v + kvo, kv_row,
                    a->out + qo);
        memcpy(slot, S, sizeof(double) * dd); /* final state of the kv head written back */
    }
    free(S);
    return NULL;
}

static int run_gqa(gqa_job_t *a)
{
    if (a->Hkv < 1 || a->H < 1 || a->H % a->Hkv != 0)
        return -1;
    int nt = a->nthreads < 1 ? 1 : a->nthreads;
    const int pairs = a->B * a->Hkv;
    if (nt > pairs)
        nt = pairs > 0 ? pairs : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
    gqa_job_t *jobs = (gqa_job_t *)malloc(sizeof(gqa_job_t) * nt);
    for (int i = 0; i < nt; i++) {
        jobs[i] = *a;
        jobs[i].nthreads = nt;
        jobs[i].tid = i;
        if (nt == 1 || pthread_create(&th[i], NULL, gqa_worker, &jobs[i]) != 0) {
            gqa_worker(&jobs[i]);
            th[i] = 0;
        }
    }
    for (int i = 0; i < nt; i++)
        if (th[i])
            pthread_join(th[i], NULL);
    free(th);
    free(jobs);
    return 0;
}

/* Packed varlen extend with grouped-query heads: q, out are [T][H*D]; k, v are [T][Hkv*D];
 * slopes [Hkv]; pool [num_slots][Hkv][D][D].  Returns -1 if H is not a multiple of Hkv. */
int la_oracle_extend_gqa(const double *q, const double *k, const double *v, const double *slopes,
                         double *pool, const int32_t *state_idx, const int32_t *cu_seqlens,
                         const uint8_t *prefix_mask, double *out, int B, int H, int Hkv, int D,
                         int nthreads)
{
    gqa_job_t a = {0};
    a.q = q; a.k = k; a.v = v; a.slopes = slopes; a.pool = pool;
    a.state_idx = state_idx; a.cu_seqlens = cu_seqlens; a.prefix_mask = prefix_mask;
    a.out = out; a.B = B; a.H = H; a.Hkv = Hkv; a.D = D; a.nthreads = nthreads;
    return run_gqa(&a);
}

/* One-token decode with grouped-query heads: q, out [B][H*D]; k, v [B][Hkv*D]. */
int la_oracle_decode_gqa(const double *q, const double *k, const double *v, const double *slopes,
                         double *pool, const int32_t *state_idx, double *out, int B, int H,
                         int Hkv, int D, int nthreads)
{
    gqa_job_t a = {0};
    a.decode = 1;
    a.q = q; a.k = k; a.v = v; a.slopes = slopes; a.pool = pool; a.state_idx = state_idx;
    a.out = out; a.B = B; a.H = H; a.Hkv = Hkv; a.D = D; a.nthreads = nthreads;
    return run_gqa(&a);
}

/* Accepted-state commit after a verify: for each request b with accept[b] >= 0, the pool slot
 * state_idx[b] takes the state after draft token accept[b] (inter[b][accept[b]], all heads);
 * accept[b] == -1 leaves the slot alone.  Returns -1 (and changes nothing) if some accept[b] is
 * outside [-1, N-1]. */
int la_oracle_commit_accepted(const double *inter, const int32_t *accept, double *pool,
                              const int32_t *state_idx, int B, int N, int H, int D)
{
    for (int b = 0; b < B; b++)
        if (accept[b] < -1 || accept[b] >= N)
            return -1;
    const size_t hdd = (size_t)H * D * D;
    for (int b = 0; b < B; b++) {
        int a = accept[b];
        if (a < 0)
            continue;
        memcpy(pool + (size_t)state_idx[b] * hdd, inter + ((size_t)b * N + a) * hdd,
               sizeof(double) * hdd);
    }
    return 0;
}
