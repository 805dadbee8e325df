/*
 * pkv_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of the decode step over a KV cache,
 * written from the pages' statement of the problem.  It exists to check the
 * CUDA path: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no code, header, table or helper with the CUDA
 * library and includes nothing from it.
 *
 * Sources followed (page title, section):
 *   [RC]  "Running Out of Cache" (serving plate XXIII.3): the cache is split
 *         into fixed blocks, a sequence's blocks need not be adjacent, and a
 *         block table maps a sequence's positions to physical blocks, the way
 *         a page table maps virtual to physical memory (paragraph "Their fix,
 *         PagedAttention ..."; Terms: "Block table", "Paged attention").
 *         Several sequences may point at the same blocks and copy only on
 *         write (section "Fragmentation is lost users").
 *   [PA]  "Efficient Memory Management for Large Language Model Serving with
 *         PagedAttention" (summary page): fixed-size, non-contiguous blocks
 *         allocated on demand; copy-on-write sharing of blocks (Summary;
 *         Key points).
 *   [VA4] "Insights into LLM Serving Systems: KV-Cache Memory Allocation
 *         Patterns", section 4, Observation-1: each decode iteration grows a
 *         request's KV by exactly one token.
 *   [VA5] "Leveraging Low-Level CUDA APIs for vAttention's Dynamic Memory",
 *         section 5.2.3: per layer, one K (or V) tensor for the maximum
 *         batch; a request's sub-tensor sits at offset reqId x S, S being the
 *         per-request maximum size.
 *
 * What is computed is the plain definition.  Paging only moves where the
 * bytes live ([RC]), so decode attention over a paged cache equals ordinary
 * single-query attention over the logical sequence that the block table
 * spells out:
 *     s_j = scale * sum_d q[d] * K[j][d]            j = 0 .. ctx-1
 *     o   = sum_j softmax(s)_j * V[j][:]
 * computed here in fp64 in two passes (max, then exponentials and sums).
 * The pages never write this formula out; it is the standard attention of
 * the models they serve, and its readings (scale, grouping of query heads
 * onto KV heads, ctx <= 0 giving zeros) are listed in the design notes.
 *
 * Layouts (our choice; the pages fix none):
 *   paged cache   [num_blocks][Hkv][bs][D]   element (b,h,o,d)
 *   contig buffer [max_reqs][Hkv][S][D]      element (r,h,p,d)
 *   q, out        [B][Hq][D];  new k, v  [T][Hkv][D]
 * bf16 values are carried as uint16_t bit patterns and widened exactly.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC -pthread
 *        pkv_oracle.c -lm   (see build_oracle.py next to this file)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 -> fp64, exact: a bf16 is the top half of an IEEE binary32. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------------- */
/* Gathers: spell out the logical K (or V) rows of one sequence, one KV    */
/* head, by following the block table [RC] or the reqId x S rule [VA5].    */
/* ---------------------------------------------------------------------- */

/* Logical row j of a paged sequence lives in physical block
 * block_table[j / bs] at in-block offset j % bs ([RC]: "a block table maps
 * positions to blocks").  Copies ctx rows of D bf16 into out[ctx][D].
 * Returns 0, or -1 if a table entry falls outside [0, num_blocks). */
int pkv_oracle_gather_paged(const uint16_t *cache, int64_t num_blocks,
                            const int32_t *block_table_row, int32_t ctx,
                            int32_t Hkv, int32_t bs, int32_t D, int32_t h,
                            uint16_t *out)
{
    for (int32_t j = 0; j < ctx; ++j) {
        int32_t logical_block = j / bs;
        int32_t offset = j % bs;
        int64_t physical = block_table_row[logical_block];
        if (physical < 0 || physical >= num_blocks)
            return -1;
        const uint16_t *row =
            cache + (((physical * Hkv + h) * (int64_t)bs + offset) * D);
        memcpy(out + (int64_t)j * D, row, (size_t)D * sizeof(uint16_t));
    }
    return 0;
}

/* Logical row j of request reqId lives at position j of that request's
 * sub-tensor, which starts at reqId x S ([VA5]).  S counts tokens. */
int pkv_oracle_gather_contig(const uint16_t *buf, int32_t max_reqs,
                             int32_t req_id, int64_t S, int32_t ctx,
                             int32_t Hkv, int32_t D, int32_t h, uint16_t *out)
{
    if (req_id < 0 || req_id >= max_reqs || (int64_t)ctx > S)
        return -1;
    for (int32_t j = 0; j < ctx; ++j) {
        const uint16_t *row =
            buf + ((((int64_t)req_id * Hkv + h) * S + j) * D);
        memcpy(out + (int64_t)j * D, row, (size_t)D * sizeof(uint16_t));
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Attention of one query over ctx gathered rows: the plain definition.    */
/* ---------------------------------------------------------------------- */

/* o[D] = sum_j softmax(scale * q.K_j)_j * V_j, all in fp64, two passes.
 * ctx <= 0 gives o = 0 (softmax over nothing is undefined; our reading). */
void pkv_oracle_attend(const uint16_t *q, const uint16_t *K, const uint16_t *V,
                       int32_t ctx, int32_t D, double scale, double *scores,
                       double *o)
{
    for (int32_t d = 0; d < D; ++d)
        o[d] = 0.0;
    if (ctx <= 0)
        return;

    /* scores s_j = scale * <q, K_j> */
    double smax = -INFINITY;
    for (int32_t j = 0; j < ctx; ++j) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += bf16_value(q[d]) * bf16_value(K[(int64_t)j * D + d]);
        scores[j] = scale * dot;
        if (scores[j] > smax)
            smax = scores[j];
    }

    /* softmax weights p_j = exp(s_j - max) / sum_k exp(s_k - max) */
    double denom = 0.0;
    for (int32_t j = 0; j < ctx; ++j) {
        scores[j] = exp(scores[j] - smax);
        denom += scores[j];
    }

    /* o = sum_j p_j V_j */
    for (int32_t j = 0; j < ctx; ++j) {
        double p = scores[j] / denom;
        for (int32_t d = 0; d < D; ++d)
            o[d] += p * bf16_value(V[(int64_t)j * D + d]);
    }
}

/* ---------------------------------------------------------------------- */
/* Whole decode batch, paged or contiguous.                                */
/* Query head h reads KV head h / (Hq / Hkv) (consecutive grouping).       */
/* Work is split over threads by (sequence, query head); each (seq, head)  */
/* is computed start to finish by one thread exactly as above.             */
/* ---------------------------------------------------------------------- */

typedef struct {
    int contig;
    const uint16_t *q, *k, *v;
    int64_t num_blocks;          /* paged: physical blocks in the cache    */
    const int32_t *block_tables; /* paged: [B][max_blocks]                 */
    int32_t max_blocks;
    int32_t bs;
    const int32_t *req_ids;      /* contig: [B]                            */
    int32_t max_reqs;
    int64_t S;
    const int32_t *context_lens;
    int32_t B, Hq, Hkv, D;
    double scale;
    double *out;                 /* [B][Hq][D]                             */
    int32_t max_ctx;
    int nthreads, tid;
    int status;
} decode_job;

static void *decode_worker(void *arg)
{
    decode_job *job = (decode_job *)arg;
    int64_t rows = job->max_ctx > 0 ? job->max_ctx : 1;
    uint16_t *K = malloc((size_t)(rows * job->D) * sizeof(uint16_t));
    uint16_t *V = malloc((size_t)(rows * job->D) * sizeof(uint16_t));
    double *scores = malloc((size_t)rows * sizeof(double));
    if (!K || !V || !scores) {
        job->status = -2;
        goto done;
    }
    int32_t group = job->Hq / job->Hkv;
    int64_t pairs = (int64_t)job->B * job->Hq;
    for (int64_t p = job->tid; p < pairs; p += job->nthreads) {
        int32_t i = (int32_t)(p / job->Hq);
        int32_t hq = (int32_t)(p % job->Hq);
        int32_t hkv = hq / group;
        int32_t ctx = job->context_lens[i];
        double *o = job->out + p * job->D;
        int rc = 0;
        if (ctx > 0) {
            if (job->contig) {
                rc |= pkv_oracle_gather_contig(job->k, job->max_reqs,
                                               job->req_ids[i], job->S, ctx,
                                               job->Hkv, job->D, hkv, K);
                rc |= pkv_oracle_gather_contig(job->v, job->max_reqs,
                                               job->req_ids[i], job->S, ctx,
                                               job->Hkv, job->D, hkv, V);
            } else {
                if ((int64_t)ctx > (int64_t)job->max_blocks * job->bs) {
                    rc = -1;
                } else {
                    const int32_t *row =
                        job->block_tables + (int64_t)i * job->max_blocks;
                    rc |= pkv_oracle_gather_paged(job->k, job->num_blocks, row,
                                                  ctx, job->Hkv, job->bs,
                                                  job->D, hkv, K);
                    rc |= pkv_oracle_gather_paged(job->v, job->num_blocks, row,
                                                  ctx, job->Hkv, job->bs,
                                                  job->D, hkv, V);
                }
            }
        }
        if (rc != 0) {
            job->status = -1;
            goto done;
        }
        pkv_oracle_attend(job->q + p * job->D, K, V, ctx, job->D, job->scale,
                          scores, o);
    }
done:
    free(K);
    free(V);
    free(scores);
    return NULL;
}

static int run_decode(decode_job *proto, int nthreads)
{
    int32_t max_ctx = 0;
    if (proto->B < 0 || proto->Hq <= 0 || proto->Hkv <= 0 || proto->D <= 0 ||
        proto->Hq % proto->Hkv != 0)
        return -3;
    for (int32_t i = 0; i < proto->B; ++i)
        if (proto->context_lens[i] > max_ctx)
            max_ctx = proto->context_lens[i];
    proto->max_ctx = max_ctx;
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    decode_job *jobs = calloc((size_t)nthreads, sizeof *jobs);
    pthread_t *th = calloc((size_t)nthreads, sizeof *th);
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -2;
    }
    int launched = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].nthreads = nthreads;
        jobs[t].tid = t;
        jobs[t].status = 0;
        if (nthreads == 1) {
            decode_worker(&jobs[t]);
        } else if (pthread_create(&th[t], NULL, decode_worker, &jobs[t]) != 0) {
            jobs[t].status = -2;
            break;
        }
        launched = t + 1;
    }
    int status = 0;
    for (int t = 0; t < launched; ++t) {
        if (nthreads > 1)
            pthread_join(th[t], NULL);
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != 0)
            status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}

/* Paged decode attention ([RC], [PA]).  out is fp64 [B][Hq][D].
 * Returns 0; -1 on a block id or context outside the table; -2 on an
 * allocation failure; -3 on bad sizes. */
int pkv_oracle_paged_decode(const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, int64_t num_blocks,
                            const int32_t *block_tables, int32_t max_blocks,
                            const int32_t *context_lens, int32_t B, int32_t Hq,
                            int32_t Hkv, int32_t D, int32_t bs, double scale,
                            double *out, int nthreads)
{
    if (bs <= 0)
        return -3;
    decode_job job;
    memset(&job, 0, sizeof job);
    job.contig = 0;
    job.q = q;
    job.k = k_cache;
    job.v = v_cache;
    job.num_blocks = num_blocks;
    job.block_tables = block_tables;
    job.max_blocks = max_blocks;
    job.bs = bs;
    job.context_lens = context_lens;
    job.B = B;
    job.Hq = Hq;
    job.Hkv = Hkv;
    job.D = D;
    job.scale = scale;
    job.out = out;
    return run_decode(&job, nthreads);
}

/* Contiguous-layout decode attention ([VA5]): request i's rows are the
 * sub-tensor of buffer row req_ids[i].  Same return codes. */
int pkv_oracle_contig_decode(const uint16_t *q, const uint16_t *k_buf,
                             const uint16_t *v_buf, const int32_t *req_ids,
                             int32_t max_reqs, const int32_t *context_lens,
                             int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                             int64_t S, double scale, double *out, int nthreads)
{
    if (S <= 0)
        return -3;
    decode_job job;
    memset(&job, 0, sizeof job);
    job.contig = 1;
    job.q = q;
    job.k = k_buf;
    job.v = v_buf;
    job.req_ids = req_ids;
    job.max_reqs = max_reqs;
    job.S = S;
    job.context_lens = context_lens;
    job.B = B;
    job.Hq = Hq;
    job.Hkv = Hkv;
    job.D = D;
    job.scale = scale;
    job.out = out;
    return run_decode(&job, nthreads);
}

/* ---------------------------------------------------------------------- */
/* Prefill over a paged cache: a chunk of new tokens per sequence, whose K  */
/* and V rows are already in the cache, attends causally.  The pages name   */
/* prefill only as a phase ([VA4], section headings); the reading here is   */
/* the standard causal one: sequence i's chunk holds the last Lq_i of its   */
/* ctx_i positions (Lq_i = cu_q[i+1] - cu_q[i]), and its j-th token, at      */
/* position ctx_i - Lq_i + j, attends positions 0 .. ctx_i - Lq_i + j.  A    */
/* chunk of one token is the decode step above.                             */
/* Work is split over threads by (token, query head); each is computed       */
/* start to finish by one thread: gather its positions, then attend.         */
/* ---------------------------------------------------------------------- */

typedef struct {
    const uint16_t *q, *k, *v;   /* q [T][Hq][D] */
    int64_t num_blocks;
    const int32_t *block_tables;
    int32_t max_blocks, bs;
    const int32_t *context_lens, *cu_q;
    int32_t B, T, Hq, Hkv, D;
    double scale;
    double *out;                 /* [T][Hq][D] */
    int32_t max_ctx;
    int nthreads, tid, status;
} prefill_job;

static void *prefill_worker(void *arg)
{
    prefill_job *job = (prefill_job *)arg;
    int64_t rows = job->max_ctx > 0 ? job->max_ctx : 1;
    uint16_t *K = malloc((size_t)(rows * job->D) * sizeof(uint16_t));
    uint16_t *V = malloc((size_t)(rows * job->D) * sizeof(uint16_t));
    double *scores = malloc((size_t)rows * sizeof(double));
    if (!K || !V || !scores) {
        job->status = -2;
        goto done;
    }
    int32_t group = job->Hq / job->Hkv;
    int64_t work = (int64_t)job->T * job->Hq;
    for (int64_t w = job->tid; w < work; w += job->nthreads) {
        int32_t t = (int32_t)(w / job->Hq);
        int32_t hq = (int32_t)(w % job->Hq);
        int32_t kv_head = hq / group;
        int32_t i = 0; /* the sequence whose chunk holds token t */
        while (i + 1 < job->B && job->cu_q[i + 1] <= t)
            ++i;
        int32_t Lq = job->cu_q[i + 1] - job->cu_q[i];
        int32_t ctx = job->context_lens[i];
        int32_t pos = ctx - Lq + (t - job->cu_q[i]);
        int32_t n = pos + 1; /* positions 0 .. pos */
        double *o = job->out + w * job->D;
        if (n <= 0 || n > ctx || (int64_t)ctx > (int64_t)job->max_blocks * job->bs) {
            job->status = -1;
            goto done;
        }
        const int32_t *row = job->block_tables + (int64_t)i * job->max_blocks;
        int rc = pkv_oracle_gather_paged(job->k, job->num_blocks, row, n, job->Hkv, job->bs,
                                         job->D, kv_head, K);
        rc |= pkv_oracle_gather_paged(job->v, job->num_blocks, row, n, job->Hkv, job->bs,
                                      job->D, kv_head, V);
        if (rc != 0) {
            job->status = -1;
            goto done;
        }
        pkv_oracle_attend(job->q + w * job->D, K, V, n, job->D, job->scale, scores, o);
    }
done:
    free(K);
    free(V);
    free(scores);
    return NULL;
}

/* Paged causal prefill.  out is fp64 [T][Hq][D], T = cu_q[B].  Returns 0;
 * -1 on a chunk longer than its context, a bad block id or a context beyond
 * the table; -2 on an allocation failure; -3 on bad sizes. */
int pkv_oracle_paged_prefill(const uint16_t *q, const uint16_t *k_cache,
                             const uint16_t *v_cache, int64_t num_blocks,
                             const int32_t *block_tables, int32_t max_blocks,
                             const int32_t *context_lens, const int32_t *cu_q,
                             int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t bs,
                             double scale, double *out, int nthreads)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || bs <= 0 || Hq % Hkv != 0 || cu_q[0] != 0)
        return -3;
    prefill_job proto;
    memset(&proto, 0, sizeof proto);
    proto.q = q;
    proto.k = k_cache;
    proto.v = v_cache;
    proto.num_blocks = num_blocks;
    proto.block_tables = block_tables;
    proto.max_blocks = max_blocks;
    proto.bs = bs;
    proto.context_lens = context_lens;
    proto.cu_q = cu_q;
    proto.B = B;
    proto.T = cu_q[B];
    proto.Hq = Hq;
    proto.Hkv = Hkv;
    proto.D = D;
    proto.scale = scale;
    proto.out = out;
    for (int32_t i = 0; i < B; ++i) {
        if (cu_q[i + 1] < cu_q[i])
            return -3;
        if (context_lens[i] > proto.max_ctx)
            proto.max_ctx = context_lens[i];
    }
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    prefill_job *jobs = calloc((size_t)nthreads, sizeof *jobs);
    pthread_t *th = calloc((size_t)nthreads, sizeof *th);
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -2;
    }
    int launched = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].nthreads = nthreads;
        jobs[t].tid = t;
        if (nthreads == 1) {
            prefill_worker(&jobs[t]);
        } else if (pthread_create(&th[t], NULL, prefill_worker, &jobs[t]) != 0) {
            jobs[t].status = -2;
            break;
        }
        launched = t + 1;
    }
    int status = 0;
    for (int t = 0; t < launched; ++t)
        if (nthreads > 1)
            pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != 0)
            status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}

/* ---------------------------------------------------------------------- */
/* KV append ([VA4] Observation-1; [RC]): the new token t's K and V rows   */
/* for every KV head go to slot_mapping[t], where a slot names physical     */
/* block slot / bs and offset slot % bs (paged), or, with bs := S, request  */
/* row slot / S and position slot % S (contiguous).  A negative slot is a   */
/* padding token and is skipped (our convention).                           */
/* Returns 0, or -1 if a slot is >= num_slots (nothing after it is written).*/
/* ---------------------------------------------------------------------- */
int pkv_oracle_kv_append(const int64_t *slot_mapping, int64_t T,
                         const uint16_t *k, const uint16_t *v,
                         uint16_t *k_cache, uint16_t *v_cache,
                         int64_t num_slots, int64_t bs, int32_t Hkv, int32_t D)
{
    if (bs <= 0)
        return -3;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots)
            return -1;
        int64_t block = slot / bs;
        int64_t offset = slot % bs;
        for (int32_t h = 0; h < Hkv; ++h) {
            int64_t dst = ((block * Hkv + h) * bs + offset) * D;
            int64_t src = (t * Hkv + h) * (int64_t)D;
            memcpy(k_cache + dst, k + src, (size_t)D * sizeof(uint16_t));
            memcpy(v_cache + dst, v + src, (size_t)D * sizeof(uint16_t));
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Copy-on-write block copy ([PA], [RC]): for every (src, dst) pair and     */
/* every layer, the whole block (all KV heads, all offsets) of K and of V   */
/* is copied from src to dst.  pairs is [n][2] int64; the caches are host   */
/* arrays of num_layers pointers.  Returns 0 or -1 on an id out of range.   */
/* ---------------------------------------------------------------------- */
int pkv_oracle_block_copy(const int64_t *pairs, int64_t n,
                          uint16_t *const *k_caches, uint16_t *const *v_caches,
                          int32_t num_layers, int64_t num_blocks,
                          int64_t block_elems)
{
    for (int64_t c = 0; c < n; ++c) {
        int64_t src = pairs[2 * c], dst = pairs[2 * c + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
            return -1;
        for (int32_t l = 0; l < num_layers; ++l) {
            memmove(k_caches[l] + dst * block_elems,
                    k_caches[l] + src * block_elems,
                    (size_t)block_elems * sizeof(uint16_t));
            memmove(v_caches[l] + dst * block_elems,
                    v_caches[l] + src * block_elems,
                    (size_t)block_elems * sizeof(uint16_t));
        }
    }
    return 0;
}
