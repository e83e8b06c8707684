/*
 * hss_oracle.c -- the CPU oracle for the high-speed-swap low-rank block predictor.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the predictor computes.  It exists so that the CUDA
 * library can be checked against something that shares no code with it.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it; the product path never does.
 *
 * Source of the method: the page "metrale_storage/predictor.rs" (module
 * docs; PredictorDims; Predictor::project_q_on_stream,
 * Predictor::project_kv_block_on_stream, Predictor::score_blocks_on_stream).
 * The tie-break rule of the victim ranking follows the page
 * "metrale_model_layers/layers/qsa_select.rs" (QsaIndexer::prefill_select,
 * host top-k: lower index first among equal scores).
 *
 * Precision points (the pages store the projections as BF16):
 *   - projections are summed in fp64 and rounded once, to the nearest bf16
 *     (ties to even), at the point where the page stores them;
 *   - scores are summed in fp64 over the bf16 values.
 * bf16 values travel as their 16-bit patterns (uint16_t).
 *
 * Every function takes plain integers and pointers; nothing here is shared
 * with the CUDA sources.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 <-> double                                                          */
/* ------------------------------------------------------------------------ */

/* Value of a bf16 bit pattern: it is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bf16, ties to even, in one step (no detour
 * through binary32, so there is no double rounding).
 *
 * bf16 keeps 8 significant bits (1 implicit + 7 stored) and the binary32
 * exponent range: normal numbers down to 2^-126, subnormals spaced 2^-133,
 * largest finite value (2 - 2^-7) * 2^127.  For |x| = m * 2^e with m in
 * [0.5, 1), the last kept bit weighs 2^(e-8); below the normal range the
 * spacing stays 2^-133.  nearbyint() rounds to nearest even under the
 * default floating-point environment.
 */
uint16_t orc_bf16_from_double(double x)
{
    float f;
    if (isnan(x)) {
        return (uint16_t)(signbit(x) ? 0xFFC0u : 0x7FC0u);
    }
    if (x == 0.0 || isinf(x)) {
        f = (float)x; /* exact, keeps the sign of zero */
    } else {
        int e;
        (void)frexp(fabs(x), &e);
        int qexp = e - 8;
        if (qexp < -133) {
            qexp = -133;
        }
        double q = nearbyint(ldexp(x, -qexp));
        double y = ldexp(q, qexp);
        if (fabs(y) > 0x1.FEp127) {
            y = copysign(INFINITY, x);
        }
        f = (float)y; /* exact: y has at most 8 significant bits */
    }
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Batch forms, used by the tests. */
void orc_bf16_from_double_n(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) {
        out[i] = orc_bf16_from_double(x[i]);
    }
}

void orc_bf16_to_double_n(const uint16_t* b, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) {
        out[i] = orc_bf16_to_double(b[i]);
    }
}

/* ------------------------------------------------------------------------ */
/* A tiny thread fan-out: run fn(ctx, i) for i in [0, n) on nthreads threads */
/* ------------------------------------------------------------------------ */

typedef void (*orc_item_fn)(void* ctx, int64_t i);

typedef struct {
    orc_item_fn fn;
    void* ctx;
    int64_t begin, end;
} orc_range;

static void* orc_range_main(void* arg)
{
    orc_range* rg = (orc_range*)arg;
    for (int64_t i = rg->begin; i < rg->end; ++i) {
        rg->fn(rg->ctx, i);
    }
    return NULL;
}

static void orc_parallel_for(int64_t n, int nthreads, orc_item_fn fn, void* ctx)
{
    if (nthreads < 1) {
        nthreads = 1;
    }
    if (nthreads > 256) {
        nthreads = 256;
    }
    if (nthreads == 1 || n < 2) {
        for (int64_t i = 0; i < n; ++i) {
            fn(ctx, i);
        }
        return;
    }
    pthread_t tid[256];
    orc_range rg[256];
    int started[256];
    int64_t chunk = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        int64_t b = (int64_t)t * chunk;
        int64_t e = b + chunk < n ? b + chunk : n;
        rg[t].fn = fn;
        rg[t].ctx = ctx;
        rg[t].begin = b < n ? b : n;
        rg[t].end = e;
        started[t] = pthread_create(&tid[t], NULL, orc_range_main, &rg[t]) == 0;
        if (!started[t]) {
            orc_range_main(&rg[t]); /* run inline if no thread could start */
        }
    }
    for (int t = 0; t < nthreads; ++t) {
        if (started[t]) {
            pthread_join(tid[t], NULL);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Step 1: query projection, Qp = Q . P  (Predictor::project_q_on_stream)   */
/* ------------------------------------------------------------------------ */

/*
 * Q  : [num_vectors, head_dim] bf16, one vector per (query row, query head);
 * P  : [head_dim, r] bf16 (row d, column j);
 * Qp : [num_vectors, r] bf16,  Qp[v][j] = bf16( sum_d Q[v][d] * P[d][j] ).
 * The page stores q_proj as BF16, so the fp64 sum is rounded once here.
 */
typedef struct {
    const uint16_t* Q;
    const uint16_t* P;
    uint16_t* Qp;
    int hd, r;
} orc_q_ctx;

static void orc_q_item(void* c, int64_t v)
{
    orc_q_ctx* k = (orc_q_ctx*)c;
    for (int j = 0; j < k->r; ++j) {
        double acc = 0.0;
        for (int d = 0; d < k->hd; ++d) {
            acc += orc_bf16_to_double(k->Q[v * k->hd + d]) *
                   orc_bf16_to_double(k->P[(int64_t)d * k->r + j]);
        }
        k->Qp[v * k->r + j] = orc_bf16_from_double(acc);
    }
}

void orc_project_q(const uint16_t* Q, int64_t num_vectors, int head_dim, const uint16_t* P,
                   int r, uint16_t* Qp, int nthreads)
{
    orc_q_ctx k = {Q, P, Qp, head_dim, r};
    orc_parallel_for(num_vectors, nthreads, orc_q_item, &k);
}

/* ------------------------------------------------------------------------ */
/* Step 2: key projection into A_g (Predictor::project_kv_block_on_stream)  */
/* ------------------------------------------------------------------------ */

/*
 * K      : [n, block_size, num_kv_heads, head_dim] bf16; entry i is the
 *          page's `k_block` ([block_size, num_kv_heads, head_dim], token-major)
 *          for the block whose id is block_ids[i];
 * A_g    : [num_layers, max_blocks, num_kv_heads, block_size, r] bf16
 *          (the per-token layout of PredictorDims::a_g_bytes);
 * result : A_g[layer][id][h][t][j] = bf16( sum_d K[i][t][h][d] * P[d][j] ).
 * Token-major input, head-major slot: the slot transposes (t, h) to (h, t).
 * Returns 0, or the 1-based position of the first block whose id lies outside
 * [0, max_blocks) (that block is skipped), or -1 if layer is out of range
 * (nothing is written), mirroring the page's range check.
 */
typedef struct {
    const uint16_t* P;
    const uint16_t* K;
    const int32_t* ids;
    uint16_t* A;
    int64_t layer, max_blocks;
    int nkv, bs, hd, r;
} orc_kv_ctx;

static void orc_kv_item(void* c, int64_t i)
{
    orc_kv_ctx* k = (orc_kv_ctx*)c;
    int64_t id = k->ids[i];
    if (id < 0 || id >= k->max_blocks) {
        return;
    }
    int64_t slot_elems = (int64_t)k->nkv * k->bs * k->r;
    uint16_t* slot = k->A + (k->layer * k->max_blocks + id) * slot_elems;
    const uint16_t* kb = k->K + i * (int64_t)k->bs * k->nkv * k->hd;
    for (int t = 0; t < k->bs; ++t) {
        for (int h = 0; h < k->nkv; ++h) {
            const uint16_t* krow = kb + ((int64_t)t * k->nkv + h) * k->hd;
            for (int j = 0; j < k->r; ++j) {
                double acc = 0.0;
                for (int d = 0; d < k->hd; ++d) {
                    acc += orc_bf16_to_double(krow[d]) *
                           orc_bf16_to_double(k->P[(int64_t)d * k->r + j]);
                }
                slot[((int64_t)h * k->bs + t) * k->r + j] = orc_bf16_from_double(acc);
            }
        }
    }
}

int64_t orc_project_kv_blocks(const uint16_t* P, const uint16_t* K, int64_t layer,
                              const int32_t* block_ids, int64_t n, int64_t num_layers,
                              int64_t max_blocks, int num_kv_heads, int block_size,
                              int head_dim, int r, uint16_t* A_g, int nthreads)
{
    if (layer < 0 || layer >= num_layers) {
        return -1;
    }
    orc_kv_ctx k = {P, K, block_ids, A_g, layer, max_blocks, num_kv_heads, block_size,
                    head_dim, r};
    orc_parallel_for(n, nthreads, orc_kv_item, &k);
    for (int64_t i = 0; i < n; ++i) {
        if (block_ids[i] < 0 || block_ids[i] >= max_blocks) {
            return i + 1;
        }
    }
    return 0;
}

/*
 * Step 2, token by token, at cache-write time (the page's per-block ingest loop,
 * Predictor::project_kv_block_on_stream, moved to where new keys are written).
 *
 * K_tok   : [n, num_kv_heads, head_dim] bf16, the layer's keys of n new tokens;
 * slots   : token i goes to block s / block_size, position s % block_size, where
 *           s = slots[i]; a negative slot marks a padding token (nothing written);
 * K_cache : [max_blocks, block_size, num_kv_heads, head_dim] bf16 or NULL; gets
 *           K_cache[blk][t][h][:] = K_tok[i][h][:] (a copy);
 * A_g     : gets A_g[layer][blk][h][t][j] = bf16( sum_d K_tok[i][h][d] * P[d][j] ).
 * Returns 0, or the 1-based position of the first token whose slot is at or
 * past max_blocks * block_size (skipped), or -1 if layer is out of range.
 */
typedef struct {
    const uint16_t* P;
    const uint16_t* K;
    const int64_t* slots;
    uint16_t* cache;
    uint16_t* A;
    int64_t layer, max_blocks;
    int nkv, bs, hd, r;
} orc_tok_ctx;

static void orc_tok_item(void* c, int64_t i)
{
    orc_tok_ctx* k = (orc_tok_ctx*)c;
    int64_t s = k->slots[i];
    if (s < 0 || s >= k->max_blocks * k->bs) {
        return;
    }
    int64_t blk = s / k->bs;
    int t = (int)(s % k->bs);
    for (int h = 0; h < k->nkv; ++h) {
        const uint16_t* krow = k->K + (i * k->nkv + h) * (int64_t)k->hd;
        if (k->cache != NULL) {
            uint16_t* crow = k->cache + ((blk * k->bs + t) * k->nkv + h) * (int64_t)k->hd;
            memcpy(crow, krow, (size_t)k->hd * sizeof(uint16_t));
        }
        uint16_t* arow = k->A + (((k->layer * k->max_blocks + blk) * k->nkv + h) * k->bs + t) *
                                    (int64_t)k->r;
        for (int j = 0; j < k->r; ++j) {
            double acc = 0.0;
            for (int d = 0; d < k->hd; ++d) {
                acc += orc_bf16_to_double(krow[d]) *
                       orc_bf16_to_double(k->P[(int64_t)d * k->r + j]);
            }
            arow[j] = orc_bf16_from_double(acc);
        }
    }
}

int64_t orc_write_kv_tokens(const uint16_t* P, const uint16_t* K_tok, const int64_t* slots,
                            int64_t n, int64_t num_layers, int64_t max_blocks, int num_kv_heads,
                            int block_size, int head_dim, int r, int64_t layer,
                            uint16_t* K_cache, uint16_t* A_g, int nthreads)
{
    if (layer < 0 || layer >= num_layers) {
        return -1;
    }
    orc_tok_ctx k = {P, K_tok, slots, K_cache, A_g, layer, max_blocks, num_kv_heads,
                     block_size, head_dim, r};
    orc_parallel_for(n, nthreads, orc_tok_item, &k);
    for (int64_t i = 0; i < n; ++i) {
        if (slots[i] >= max_blocks * block_size) {
            return i + 1;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 3: block scores (Predictor::score_blocks_on_stream)                  */
/* ------------------------------------------------------------------------ */

/*
 * Qp          : [num_seqs, rows_per_seq, num_q_heads, r] bf16;
 * A_g         : as above;
 * seq_offsets : [num_seqs + 1], sequence s owns table entries
 *               [seq_offsets[s], seq_offsets[s+1]);
 * block_table : physical block id of each entry;
 * score[i]    : max over query heads h, query rows and tokens t of the block
 *               of  sum_j Qp[s][row][h][j] * A_g[layer][id][h / g][t][j],
 *               g = num_q_heads / num_kv_heads (query head h reads kv head
 *               h / g), summed in fp64;
 * tsum[i]     : for the same candidates, the largest sum_j |Qp_j * A_j|
 *               (the scale the score tolerance is measured against).
 * An entry whose id lies outside [0, max_blocks) is not scored: its score is
 * +inf, so it is never chosen as a victim, and tsum is 0.
 * Returns the number of such entries.
 */
typedef struct {
    const uint16_t* Qp;
    const uint16_t* A;
    int64_t layer, max_blocks;
    int rows, nq, nkv, r, bs;
} orc_score_shape;

/* Score one table entry of sequence s whose physical block id is id. */
static void orc_score_one(const orc_score_shape* k, int64_t s, int64_t id, double* score,
                          double* tsum)
{
    if (id < 0 || id >= k->max_blocks) {
        *score = INFINITY;
        *tsum = 0.0;
        return;
    }
    int g = k->nq / k->nkv;
    int64_t slot_elems = (int64_t)k->nkv * k->bs * k->r;
    const uint16_t* slot = k->A + (k->layer * k->max_blocks + id) * slot_elems;
    double best = -INFINITY;
    double best_abs = 0.0;
    for (int row = 0; row < k->rows; ++row) {
        for (int h = 0; h < k->nq; ++h) {
            const uint16_t* q = k->Qp + ((s * k->rows + row) * (int64_t)k->nq + h) * k->r;
            int c_kv = h / g;
            for (int t = 0; t < k->bs; ++t) {
                const uint16_t* a = slot + ((int64_t)c_kv * k->bs + t) * k->r;
                double dot = 0.0, mag = 0.0;
                for (int j = 0; j < k->r; ++j) {
                    double term = orc_bf16_to_double(q[j]) * orc_bf16_to_double(a[j]);
                    dot += term;
                    mag += fabs(term);
                }
                if (dot > best) {
                    best = dot;
                }
                if (mag > best_abs) {
                    best_abs = mag;
                }
            }
        }
    }
    *score = best;
    *tsum = best_abs;
}

typedef struct {
    orc_score_shape shape;
    const int32_t* table;
    const int64_t* seq_of_entry;
    double* score;
    double* tsum;
} orc_score_ctx;

static void orc_score_item(void* c, int64_t i)
{
    orc_score_ctx* k = (orc_score_ctx*)c;
    orc_score_one(&k->shape, k->seq_of_entry[i], k->table[i], &k->score[i], &k->tsum[i]);
}

int64_t orc_score_blocks(const uint16_t* Qp, int64_t num_seqs, int rows_per_seq,
                         int num_q_heads, int num_kv_heads, int r, int block_size,
                         const uint16_t* A_g, int64_t layer, int64_t max_blocks,
                         const int32_t* block_table, const int64_t* seq_offsets, double* score,
                         double* tsum, int nthreads)
{
    int64_t total = seq_offsets[num_seqs];
    int64_t* seq_of_entry = (int64_t*)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
    if (seq_of_entry == NULL) {
        return -1;
    }
    for (int64_t s = 0; s < num_seqs; ++s) {
        for (int64_t i = seq_offsets[s]; i < seq_offsets[s + 1]; ++i) {
            seq_of_entry[i] = s;
        }
    }
    orc_score_ctx k;
    k.shape.Qp = Qp;
    k.shape.A = A_g;
    k.shape.layer = layer;
    k.shape.max_blocks = max_blocks;
    k.shape.rows = rows_per_seq;
    k.shape.nq = num_q_heads;
    k.shape.nkv = num_kv_heads;
    k.shape.r = r;
    k.shape.bs = block_size;
    k.table = block_table;
    k.seq_of_entry = seq_of_entry;
    k.score = score;
    k.tsum = tsum;
    orc_parallel_for(total, nthreads, orc_score_item, &k);
    free(seq_of_entry);
    int64_t bad = 0;
    for (int64_t i = 0; i < total; ++i) {
        if (block_table[i] < 0 || block_table[i] >= max_blocks) {
            ++bad;
        }
    }
    return bad;
}

/* Scores of a sample of table entries only (for checks at full size). */
int64_t orc_score_entries(const uint16_t* Qp, int64_t num_seqs, int rows_per_seq,
                          int num_q_heads, int num_kv_heads, int r, int block_size,
                          const uint16_t* A_g, int64_t layer, int64_t max_blocks,
                          const int32_t* block_table, const int64_t* seq_offsets,
                          const int64_t* entries, int64_t num_entries, double* score,
                          double* tsum)
{
    orc_score_shape shape;
    shape.Qp = Qp;
    shape.A = A_g;
    shape.layer = layer;
    shape.max_blocks = max_blocks;
    shape.rows = rows_per_seq;
    shape.nq = num_q_heads;
    shape.nkv = num_kv_heads;
    shape.r = r;
    shape.bs = block_size;
    int64_t bad = 0;
    for (int64_t e = 0; e < num_entries; ++e) {
        int64_t i = entries[e];
        int64_t s = 0;
        while (s + 1 < num_seqs && seq_offsets[s + 1] <= i) {
            ++s;
        }
        orc_score_one(&shape, s, block_table[i], &score[e], &tsum[e]);
        if (block_table[i] < 0 || block_table[i] >= max_blocks) {
            ++bad;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Step 3b: block scores with a valid-length mask and a causal mask          */
/* ------------------------------------------------------------------------ */

/*
 * The same score as orc_score_blocks, restricted to the visible candidates.
 * Token t of the block at table position j of sequence s (j counted from the
 * sequence's first entry) sits at position p = j * block_size + t.
 *   ctx_len  (NULL: no length mask)  token p is scored only if p < ctx_len[s];
 *   row_pos0 (NULL: no causal mask)  query row `row` sees token p only if
 *                                    p <= row_pos0[s] + row.
 * A block with no visible candidate scores -inf (tsum 0); an out-of-range id
 * still scores +inf.
 */
static void orc_score_one_masked(const orc_score_shape* k, int64_t s, int64_t id, int64_t j,
                                 const int64_t* ctx_len, const int64_t* row_pos0, double* score,
                                 double* tsum)
{
    if (id < 0 || id >= k->max_blocks) {
        *score = INFINITY;
        *tsum = 0.0;
        return;
    }
    int g = k->nq / k->nkv;
    int64_t slot_elems = (int64_t)k->nkv * k->bs * k->r;
    const uint16_t* slot = k->A + (k->layer * k->max_blocks + id) * slot_elems;
    double best = -INFINITY;
    double best_abs = 0.0;
    for (int row = 0; row < k->rows; ++row) {
        for (int h = 0; h < k->nq; ++h) {
            const uint16_t* q = k->Qp + ((s * k->rows + row) * (int64_t)k->nq + h) * k->r;
            int c_kv = h / g;
            for (int t = 0; t < k->bs; ++t) {
                int64_t pos = j * k->bs + t;
                if (ctx_len != NULL && pos >= ctx_len[s]) {
                    continue;
                }
                if (row_pos0 != NULL && pos > row_pos0[s] + row) {
                    continue;
                }
                const uint16_t* a = slot + ((int64_t)c_kv * k->bs + t) * k->r;
                double dot = 0.0, mag = 0.0;
                for (int jj = 0; jj < k->r; ++jj) {
                    double term = orc_bf16_to_double(q[jj]) * orc_bf16_to_double(a[jj]);
                    dot += term;
                    mag += fabs(term);
                }
                if (dot > best) {
                    best = dot;
                }
                if (mag > best_abs) {
                    best_abs = mag;
                }
            }
        }
    }
    *score = best;
    *tsum = best_abs;
}

typedef struct {
    orc_score_shape shape;
    const int32_t* table;
    const int64_t* seq_of_entry;
    const int64_t* seq_offsets;
    const int64_t* ctx_len;
    const int64_t* row_pos0;
    double* score;
    double* tsum;
} orc_masked_ctx;

static void orc_masked_item(void* c, int64_t i)
{
    orc_masked_ctx* k = (orc_masked_ctx*)c;
    int64_t s = k->seq_of_entry[i];
    orc_score_one_masked(&k->shape, s, k->table[i], i - k->seq_offsets[s], k->ctx_len, k->row_pos0,
                         &k->score[i], &k->tsum[i]);
}

int64_t orc_score_blocks_masked(const uint16_t* Qp, int64_t num_seqs, int rows_per_seq,
                                int num_q_heads, int num_kv_heads, int r, int block_size,
                                const uint16_t* A_g, int64_t layer, int64_t max_blocks,
                                const int32_t* block_table, const int64_t* seq_offsets,
                                const int64_t* ctx_len, const int64_t* row_pos0, double* score,
                                double* tsum, int nthreads)
{
    int64_t total = seq_offsets[num_seqs];
    int64_t* seq_of_entry = (int64_t*)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
    if (seq_of_entry == NULL) {
        return -1;
    }
    for (int64_t s = 0; s < num_seqs; ++s) {
        for (int64_t i = seq_offsets[s]; i < seq_offsets[s + 1]; ++i) {
            seq_of_entry[i] = s;
        }
    }
    orc_masked_ctx k;
    k.shape.Qp = Qp;
    k.shape.A = A_g;
    k.shape.layer = layer;
    k.shape.max_blocks = max_blocks;
    k.shape.rows = rows_per_seq;
    k.shape.nq = num_q_heads;
    k.shape.nkv = num_kv_heads;
    k.shape.r = r;
    k.shape.bs = block_size;
    k.table = block_table;
    k.seq_of_entry = seq_of_entry;
    k.seq_offsets = seq_offsets;
    k.ctx_len = ctx_len;
    k.row_pos0 = row_pos0;
    k.score = score;
    k.tsum = tsum;
    orc_parallel_for(total, nthreads, orc_masked_item, &k);
    free(seq_of_entry);
    int64_t bad = 0;
    for (int64_t i = 0; i < total; ++i) {
        if (block_table[i] < 0 || block_table[i] >= max_blocks) {
            ++bad;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Step 4: eviction victims (ascending score; lower index first on ties)    */
/* ------------------------------------------------------------------------ */

typedef struct {
    double v;
    int32_t idx;
} orc_keyed;

static int orc_keyed_cmp(const void* a, const void* b)
{
    const orc_keyed* x = (const orc_keyed*)a;
    const orc_keyed* y = (const orc_keyed*)b;
    if (x->v < y->v) {
        return -1;
    }
    if (x->v > y->v) {
        return 1;
    }
    return (x->idx > y->idx) - (x->idx < y->idx);
}

/*
 * scores      : [total] f32, the block scores in table order;
 * seq_offsets : [num_seqs + 1];
 * victims     : [num_seqs, k] int32.  Row s lists the min(k, n_s) entries of
 *               sequence s with the smallest (score, index), in ascending
 *               order, as indices into that sequence's own table
 *               (0 .. n_s - 1); the rest of the row is -1.
 * -0 compares equal to +0 and NaN is treated as +inf, so every key is totally
 * ordered and equal scores fall back to the lower index.
 */
int orc_rank_victims(const float* scores, const int64_t* seq_offsets, int64_t num_seqs, int k,
                     int32_t* victims)
{
    for (int64_t s = 0; s < num_seqs; ++s) {
        int64_t base = seq_offsets[s];
        int64_t n = seq_offsets[s + 1] - base;
        orc_keyed* keyed = (orc_keyed*)malloc(sizeof(orc_keyed) * (size_t)(n > 0 ? n : 1));
        if (keyed == NULL) {
            return -1;
        }
        for (int64_t i = 0; i < n; ++i) {
            double v = (double)scores[base + i];
            if (isnan(v)) {
                v = INFINITY;
            }
            if (v == 0.0) {
                v = 0.0; /* -0 -> +0 */
            }
            keyed[i].v = v;
            keyed[i].idx = (int32_t)i;
        }
        qsort(keyed, (size_t)n, sizeof(orc_keyed), orc_keyed_cmp);
        for (int j = 0; j < k; ++j) {
            victims[s * (int64_t)k + j] = j < n ? keyed[j].idx : -1;
        }
        free(keyed);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 5: per-row scores and per-row selection (QSA-style, page            */
/* "metrale_model_layers/layers/qsa_select.rs", host top-k per row)          */
/* ------------------------------------------------------------------------ */

/*
 * One sequence's chunk of query rows, each row on its own:
 * Qp     : [rows, num_q_heads, r] bf16;
 * table  : [n] physical block ids of the sequence, in order;
 * score[row * n + j] : max over query heads h and tokens t of block table[j]
 *          of sum_k Qp[row][h][k] * A_g[layer][table[j]][h / g][t][k], in fp64
 *          (the block score of orc_score_blocks, without the max over rows);
 * tsum   : the largest sum_k |Qp_k * A_k| over the same candidates.
 * An id outside [0, max_blocks) scores -inf (it is never selected), tsum 0.
 * Returns the number of such entries.
 */
typedef struct {
    orc_score_shape shape;
    const int32_t* table;
    int64_t n;
    double* score;
    double* tsum;
} orc_rows_ctx;

static void orc_rows_item(void* c, int64_t i)
{
    orc_rows_ctx* k = (orc_rows_ctx*)c;
    int64_t row = i / k->n;
    int64_t j = i - row * k->n;
    int64_t id = k->table[j];
    if (id < 0 || id >= k->shape.max_blocks) {
        k->score[i] = -INFINITY;
        k->tsum[i] = 0.0;
        return;
    }
    /* A one-row view of the chunk: sequence `row`, one row per sequence. */
    orc_score_shape one = k->shape;
    one.rows = 1;
    orc_score_one(&one, row, id, &k->score[i], &k->tsum[i]);
}

int64_t orc_score_rows(const uint16_t* Qp, int64_t rows, int num_q_heads, int num_kv_heads,
                       int r, int block_size, const uint16_t* A_g, int64_t layer,
                       int64_t max_blocks, const int32_t* table, int64_t n, double* score,
                       double* tsum, int nthreads)
{
    orc_rows_ctx k;
    k.shape.Qp = Qp;
    k.shape.A = A_g;
    k.shape.layer = layer;
    k.shape.max_blocks = max_blocks;
    k.shape.rows = 1;
    k.shape.nq = num_q_heads;
    k.shape.nkv = num_kv_heads;
    k.shape.r = r;
    k.shape.bs = block_size;
    k.table = table;
    k.n = n;
    k.score = score;
    k.tsum = tsum;
    orc_parallel_for(rows * n, nthreads, orc_rows_item, &k);
    int64_t bad = 0;
    for (int64_t j = 0; j < n; ++j) {
        if (table[j] < 0 || table[j] >= max_blocks) {
            ++bad;
        }
    }
    return bad;
}

/*
 * scores : [rows, stride] f32; row r's score of block j is scores[r * stride + j];
 * row r (at position first_pos + r) considers the blocks it has seen whole,
 *   j < complete_r = min(n, (first_pos + r + 1) / block_size),
 * orders them by score, larger first, lower index first among equal scores
 * (-0 equals +0; NaN ranks below every number), and lists the first topk:
 * lists[r * topk + i], -1 where complete_r <= i.
 */
int orc_select_rows(const float* scores, int64_t rows, int64_t n, int64_t stride,
                    int64_t first_pos, int block_size, int topk, int32_t* lists)
{
    orc_keyed* keyed = (orc_keyed*)malloc(sizeof(orc_keyed) * (size_t)(n > 0 ? n : 1));
    if (keyed == NULL) {
        return -1;
    }
    for (int64_t r = 0; r < rows; ++r) {
        int64_t complete = (first_pos + r + 1) / block_size;
        if (complete > n) {
            complete = n;
        }
        if (complete < 0) {
            complete = 0;
        }
        for (int64_t j = 0; j < complete; ++j) {
            double v = (double)scores[r * stride + j];
            /* ascending order of v = descending order of the score */
            v = isnan(v) ? INFINITY : -v;
            if (v == 0.0) {
                v = 0.0; /* -0 -> +0 */
            }
            keyed[j].v = v;
            keyed[j].idx = (int32_t)j;
        }
        qsort(keyed, (size_t)complete, sizeof(orc_keyed), orc_keyed_cmp);
        for (int i = 0; i < topk; ++i) {
            lists[r * (int64_t)topk + i] = i < complete ? keyed[i].idx : -1;
        }
    }
    free(keyed);
    return 0;
}
