/*
 * hss.h -- C ABI of the GB300 (sm_103a) low-rank KV-block predictor.
 *
 * The predictor ("high-speed swap" block predictor, page
 * "metrale_storage/predictor.rs", module docs) keeps, for every key token of
 * every paged KV block, a low-rank copy of the key:
 *
 *     A_g[layer][block][kv_head][token][j] = bf16( sum_d K[token][kv_head][d] * P[d][j] )
 *
 * and scores each block against the current queries as the largest projected
 * dot product Qp . A_g over query heads, query rows and the block's tokens.
 * The lowest-scoring blocks are the eviction victims.
 *
 * Conventions for every call:
 *   - bf16 tensors are passed as uint16_t bit patterns (IEEE binary32 upper
 *     halves); every tensor is dense, row-major, in the layout stated.
 *   - Pointers marked "device" must point to memory of the current CUDA
 *     device; the caller owns every buffer.  The library allocates no memory
 *     and keeps no state between calls other than the per-device kernel set-up
 *     done on first use and one device-resident error word (see
 *     hss_read_device_error).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     compute call only validates its arguments on the host and enqueues work
 *     on that stream; it returns before the work is done.  Nothing is enqueued
 *     when a call returns an error.
 *   - Argument errors are reported synchronously by the return value.  Errors
 *     that depend on device-resident data (a block id out of range) are
 *     reported through the optional `dev_status` word (device int32): the
 *     kernel stores the first error code into it if it is still HSS_OK; the
 *     caller zeroes it before the call and reads it after synchronising.
 */
#ifndef HSS_H
#define HSS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The seven predictor dimensions (PredictorDims on the predictor page).
 * num_q_heads must be a multiple of num_kv_heads (PredictorDims::validate);
 * query head h reads kv head h / (num_q_heads / num_kv_heads).
 * Shapes the kernels support: head_dim in {64, 128, 192, 256}; r in {16, 32, 64, 128};
 * block_size a multiple of 16 in [16, 256] (the tensor-core scorer: 16 or 32);
 * num_kv_heads <= 64; max_blocks <= 2^31 - 1. */
typedef struct hss_dims {
    int32_t num_layers;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t r;
    int32_t block_size;
    int64_t max_blocks;
} hss_dims;

typedef enum hss_status {
    HSS_OK = 0,
    HSS_ERR_INVALID_DIMS = 1,        /* a dimension is <= 0, or num_q_heads % num_kv_heads != 0 */
    HSS_ERR_OUT_OF_RANGE = 2,        /* layer >= num_layers, or a block id outside [0, max_blocks) */
    HSS_ERR_NULL_POINTER = 3,        /* a required pointer is NULL */
    HSS_ERR_MISALIGNED = 4,          /* a bf16 tensor is not 16-byte aligned */
    HSS_ERR_WORKSPACE_TOO_SMALL = 5, /* a caller workspace (hss_layer_step) or the static
                                        array (hss_layer_step_static) is too small */
    HSS_ERR_UNSUPPORTED_SHAPE = 6,   /* valid dims that no kernel here handles */
    HSS_ERR_CUDA = 7,                /* a CUDA runtime call or a launch failed */
    HSS_ERR_DEVICE_TIMEOUT = 8,      /* a kernel gave up waiting on a pipeline barrier */
    HSS_ERR_INVALID_ARGUMENT = 9     /* a count or size is negative or inconsistent */
} hss_status;

/* Human-readable name of a status code (static storage; never NULL). */
const char* hss_status_string(int32_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t hss_version(void);

/* HSS_OK if the dims are valid (PredictorDims::validate) and supported. */
hss_status hss_validate_dims(const hss_dims* dims);

/* Bytes of the per-token low-rank key store A_g,
 * num_layers * max_blocks * num_kv_heads * block_size * r * 2
 * (PredictorDims::a_g_bytes, predictor page); 0 if dims is NULL or invalid. */
size_t hss_a_g_bytes(const hss_dims* dims);

/*
 * Query projection: Qp = Q . P, rounded once to bf16 (round to nearest even).
 * Page "metrale_storage/predictor.rs", Predictor::project_q ("q_proj = q @ P";
 * q is [num_q_heads, head_dim] BF16, q_proj [num_q_heads, r] BF16), extended
 * here to many query rows.
 *
 *   P    device, [head_dim, r] bf16, 16-byte aligned
 *   Q    device, [num_rows, num_q_heads, head_dim] bf16, 16-byte aligned
 *   Qp   device, [num_rows, num_q_heads, r] bf16, 16-byte aligned (output)
 *   num_rows >= 0 query rows (num_rows = 0 enqueues nothing)
 * Accumulation is fp32 on the tensor cores.
 */
hss_status hss_project_q(const hss_dims* dims, const uint16_t* P, const uint16_t* Q,
                         int64_t num_rows, uint16_t* Qp, void* stream);

/*
 * Key projection of whole blocks into A_g:
 *   A_g[layer][block_ids[i]][h][t][j] = bf16( sum_d K[i][t][h][d] * P[d][j] ).
 * Page "metrale_storage/predictor.rs", Predictor::project_kv_block (k_block is
 * [block_size, num_kv_heads, head_dim] BF16, token-major; the A_g slot is
 * [num_kv_heads, block_size, r], head-major; an out-of-range layer or block
 * is an error), batched here over num_blocks blocks per call.
 *
 *   P          device, [head_dim, r] bf16, 16-byte aligned
 *   K          device, [num_blocks, block_size, num_kv_heads, head_dim] bf16,
 *              16-byte aligned
 *   layer      0 <= layer < num_layers, else HSS_ERR_OUT_OF_RANGE
 *   block_ids  device, [num_blocks] int32; ids should be distinct (two
 *              entries with the same id race for the slot).  An id outside
 *              [0, max_blocks) is skipped and sets *dev_status to
 *              HSS_ERR_OUT_OF_RANGE.
 *   A_g        device, [num_layers, max_blocks, num_kv_heads, block_size, r]
 *              bf16, 16-byte aligned; only the addressed slots are written
 *   dev_status device int32 or NULL
 */
hss_status hss_project_kv_blocks(const hss_dims* dims, const uint16_t* P, const uint16_t* K,
                                 int32_t layer, const int32_t* block_ids, int64_t num_blocks,
                                 uint16_t* A_g, int32_t* dev_status, void* stream);

/*
 * Cache write with projection: the page's ingest (Predictor::project_kv_block, launched once
 * per block after a block is written) moved to where the layer's new keys are written, one
 * token at a time.  For every token i with slot s = slots[i] = block * block_size + t:
 *   K_cache[s / block_size][s % block_size][h][:] = K_tok[i][h][:]        (if K_cache != NULL)
 *   A_g[layer][s / block_size][h][s % block_size][:] = bf16(K_tok[i][h] . P)
 * for every kv head h, in one launch.  A decode step (one new token per sequence) thus keeps
 * A_g current without waiting for a block to fill; the rows of positions not yet written
 * keep what they held (score such blocks with a ctx_len mask, hss_score_blocks_masked).
 *   K_tok    device, [num_tokens, num_kv_heads, head_dim] bf16, 16-byte aligned: the layer's
 *            keys of the new tokens
 *   slots    device, [num_tokens] int64, 8-byte aligned.  A negative slot marks a padding
 *            token: nothing is written for it.  A slot >= max_blocks * block_size is skipped
 *            and raises HSS_ERR_OUT_OF_RANGE in *dev_status (if not NULL) and the library's
 *            device error word.  If two tokens name one slot, either may win.
 *   K_cache  device, [max_blocks, block_size, num_kv_heads, head_dim] bf16, 16-byte aligned:
 *            this layer's paged key cache (each block in the page's k_block layout), or NULL
 *            to write A_g only
 *   A_g      as in hss_project_kv_blocks
 * Each A_g row equals what hss_project_kv_blocks writes for that position (the same kernel
 * computes it).  Errors as hss_project_kv_blocks.
 */
hss_status hss_write_kv_tokens(const hss_dims* dims, const uint16_t* P, const uint16_t* K_tok,
                               const int64_t* slots, int64_t num_tokens, uint16_t* K_cache,
                               uint16_t* A_g, int32_t layer, int32_t* dev_status, void* stream);

/* Score kernel choice for hss_score_blocks. */
#define HSS_PATH_AUTO 0    /* decode kernel when rows_per_seq * (num_q_heads/num_kv_heads) <= 16,
                              else the tensor-memory (tcgen05) kernel */
#define HSS_PATH_DECODE 1  /* streaming kernel: warp-level MMA per block, A_g read once */
#define HSS_PATH_TCGEN05 2 /* dense kernel for prefill chunks: tcgen05 MMA, TMEM accumulators */

/*
 * Block scores:
 *   scores[i] = max over query rows, query heads h and tokens t of block
 *               block_table[i] of  sum_j Qp[s][row][h][j] * A_g[layer][block_table[i]][h/g][t][j]
 * for i in sequence s (seq_offsets[s] <= i < seq_offsets[s+1]), g =
 * num_q_heads / num_kv_heads.  No scaling, no masking: every token of the
 * block is scored.  Page "metrale_storage/predictor.rs",
 * Predictor::score_blocks (the max over query heads and tokens of the
 * projected dot product, f32 out); that call scores contiguous slots, which
 * an identity table reproduces.
 *
 *   Qp           device, [num_seqs, rows_per_seq, num_q_heads, r] bf16,
 *                16-byte aligned
 *   rows_per_seq >= 1 query rows per sequence
 *   A_g          device, as in hss_project_kv_blocks
 *   block_table  device, [total_blocks] int32 physical block ids
 *   seq_offsets  device, [num_seqs + 1] int32, non-decreasing,
 *                seq_offsets[0] = 0, seq_offsets[num_seqs] = total_blocks
 *   scores       device, [total_blocks] f32 (output)
 *   path         HSS_PATH_*
 *   dev_status   device int32 or NULL.  A table entry outside
 *                [0, max_blocks) gets score +inf (so it is never a victim)
 *                and sets HSS_ERR_OUT_OF_RANGE.
 * Accumulation is fp32; the result differs from an exact sum by at most
 * about r * 2^-23 * sum_j |Qp_j * A_j|.
 */
hss_status hss_score_blocks(const hss_dims* dims, const uint16_t* Qp, int32_t rows_per_seq,
                            const uint16_t* A_g, int32_t layer, const int32_t* block_table,
                            const int32_t* seq_offsets, int32_t num_seqs, int64_t total_blocks,
                            float* scores, int32_t path, int32_t* dev_status, void* stream);

/*
 * Block scores restricted to visible tokens: hss_score_blocks with two optional masks.
 * Token t of the entry at table position j of sequence s (j counted from seq_offsets[s])
 * sits at position p = j * block_size + t.
 *   ctx_len   device, [num_seqs] int32, or NULL: only tokens with p < ctx_len[s] count
 *             (the tail of a partly filled last block, or blocks past the context);
 *   row_pos0  device, [num_seqs] int32, or NULL: causal mask for a chunk of query rows
 *             whose first row sits at row_pos0[s]; row r sees only p <= row_pos0[s] + r.
 * A block with no visible candidate scores -inf.  Both NULL: exactly hss_score_blocks.
 * The predictor page's scorer takes no lengths or positions (Predictor::score_blocks);
 * these masks are the next step it leaves open.  Seeing a key only from rows at or after
 * its position follows the complete-block count of "metrale_model_layers/layers/
 * qsa_select.rs" (QsaIndexer::prefill_select).
 */
hss_status hss_score_blocks_masked(const hss_dims* dims, const uint16_t* Qp, int32_t rows_per_seq,
                                   const uint16_t* A_g, int32_t layer, const int32_t* block_table,
                                   const int32_t* seq_offsets, int32_t num_seqs,
                                   int64_t total_blocks, const int32_t* ctx_len,
                                   const int32_t* row_pos0, float* scores, int32_t path,
                                   int32_t* dev_status, void* stream);

/* Largest k that hss_rank_victims accepts. */
#define HSS_MAX_VICTIMS 8192

/*
 * Eviction victims: for each sequence s, the min(k, n_s) table entries with
 * the smallest scores, in ascending order of (score, entry index), written as
 * indices into that sequence's own table (0 .. n_s - 1); the rest of the row
 * is -1.  -0 ranks equal to +0; NaN ranks as +inf.  The predictor page says
 * the scores serve only to rank eviction victims (module docs of
 * "metrale_storage/predictor.rs"); the lower-index-first rule for equal scores
 * mirrors the host top-k of "metrale_model_layers/layers/qsa_select.rs".
 *
 *   scores       device, [total_blocks] f32
 *   seq_offsets  device, [num_seqs + 1] int32, as in hss_score_blocks
 *   k            1 <= k <= HSS_MAX_VICTIMS
 *   victims      device, [num_seqs, k] int32 (output)
 * The result is exact (integer output, no tolerance).
 */
hss_status hss_rank_victims(const float* scores, const int32_t* seq_offsets, int32_t num_seqs,
                            int64_t total_blocks, int32_t k, int32_t* victims, void* stream);

/*
 * Per-row block scores (QSA-style selection, the host top-k of the page
 * "metrale_model_layers/layers/qsa_select.rs" done on the GPU, with this predictor's score):
 * for one sequence's chunk of query rows, each row on its own,
 *   scores[row * num_blocks + j] = max over query heads h and the tokens t of block
 *       block_table[j] of  sum_k Qp[row][h][k] * A_g[layer][block_table[j]][h / g][t][k]
 * i.e. the block score of hss_score_blocks without the max over rows.  Runs on the tcgen05
 * scorer (the dense prefill contraction).
 *   Qp           device, [rows, num_q_heads, r] bf16, 16-byte aligned
 *   block_table  device, [num_blocks] int32: the sequence's physical block ids, in order
 *   scores       device, [rows, num_blocks] f32 (output)
 * Supported: g = num_q_heads / num_kv_heads in {1, 2, 4, 8, 16}, block_size 16 or 32, and
 * the tcgen05 scorer's shapes; otherwise HSS_ERR_UNSUPPORTED_SHAPE.  An id outside
 * [0, max_blocks) scores -inf in every row (never selected) and raises HSS_ERR_OUT_OF_RANGE
 * in *dev_status (if not NULL) and the library's device error word.
 */
hss_status hss_score_rows(const hss_dims* dims, const uint16_t* Qp, int32_t rows,
                          const uint16_t* A_g, int32_t layer, const int32_t* block_table,
                          int64_t num_blocks, float* scores, int32_t* dev_status, void* stream);

/*
 * Per-row top-k selection (the host top-k per row of the page
 * "metrale_model_layers/layers/qsa_select.rs", QsaIndexer::prefill_select, on the GPU).
 * Row r of a prefill chunk whose first row sits at position first_pos has seen the blocks
 *   j < complete_r = min(num_blocks, (first_pos + r + 1) / block_size)
 * whole; its list holds the topk of them with the largest scores[r * num_blocks + j],
 * larger first, the lower index first among equal scores (-0 equals +0; NaN ranks like
 * -inf, below every number), as indices j; lists[r * topk + i] = -1 where i >= complete_r.
 *   scores  device, [rows, num_blocks] f32 (e.g. from hss_score_rows)
 *   lists   device, [rows, topk] int32 (output); 1 <= topk <= HSS_MAX_VICTIMS
 * The result is exact (integer output).
 */
hss_status hss_select_rows(const float* scores, int32_t rows, int64_t num_blocks,
                           int64_t first_pos, int32_t block_size, int32_t topk, int32_t* lists,
                           void* stream);

/*
 * One predictor layer call in as few launches as the shape allows: project the newly
 * written blocks into A_g and the query rows into Qp (one launch), score every table
 * entry, and rank the victims of every sequence.  Results are the same as
 *   hss_project_kv_blocks(K_new, new_ids) ; hss_project_q(Q) ; hss_score_blocks(path AUTO) ;
 *   hss_rank_victims
 * on the same stream (the same kernels compute them; the victims are the same words in
 * the same order).  In the decode regime the victim ranking runs inside the scoring kernel:
 * for at most 8 sequences and 4096 blocks in all, when the scoring grid fits on the GPU at
 * once, every CTA publishes its blocks' keys in the workspace, waits until all the call's
 * keys are there (a bounded wait: HSS_ERR_DEVICE_TIMEOUT after 1 s) and places its own blocks
 * by counting the smaller (sequence, score, position) words; otherwise the last CTA to finish
 * a sequence ranks it.  That bounded wait assumes the scoring grid gets the whole GPU: a kernel of
 * another stream that holds SMs for longer than the limit makes the call report
 * HSS_ERR_DEVICE_TIMEOUT (its victims are then wrong; zero the workspace before the next call).
 * This is the fused decode call the predictor page's per-step usage implies (module docs
 * of "metrale_storage/predictor.rs": scores only rank eviction victims).
 *
 *   K_new, new_ids, num_new  blocks written this step (num_new may be 0), as in
 *                            hss_project_kv_blocks
 *   Q                        device, [num_seqs, rows_per_seq, num_q_heads, head_dim] bf16
 *   Qp                       device, [num_seqs, rows_per_seq, num_q_heads, r] bf16 (output),
 *                            or NULL when the caller does not need the projected queries.
 *                            With NULL, the decode scorer projects the queries itself (into
 *                            shared memory; Qp is never stored), so the scoring path has one
 *                            launch fewer: only the new blocks are projected before it, and it
 *                            waits for that projection only where it reads a new block.  NULL
 *                            is accepted when the call takes the decode scorer (rows_per_seq *
 *                            num_q_heads / num_kv_heads <= 16), num_seqs <= 8, and the query
 *                            rows, P and the projected fragments fit the scorer's 96 KiB of
 *                            shared memory (the Llama-3-8B-like decode layer, 32 q / 8 kv
 *                            heads, head_dim 128, r 32, one row, needs 22 KiB); otherwise the
 *                            call returns HSS_ERR_NULL_POINTER.  The scores then come from
 *                            the same fp32-accumulated, bf16-rounded Qp, summed in another
 *                            order, so a Qp element may differ from hss_project_q's by one
 *                            bf16 ulp.
 *   scores, victims          outputs, as in hss_score_blocks / hss_rank_victims
 *   workspace                device, >= hss_layer_step_workspace_bytes(num_seqs) bytes,
 *                            4-byte aligned (16-byte aligned for the in-kernel ranking of
 *                            at most 8 sequences above): that ranking's call number and 32 KiB of
 *                            tagged keys (33024 bytes), then the per-sequence completion
 *                            counters, so calls with different num_seqs may share one
 *                            workspace sized for the largest.  Zero all of it once
 *                            (e.g. cudaMemsetAsync) before its first use, then leave it as
 *                            each call leaves it: the counters return to zero, the call
 *                            number and the keys carry over to the next call (zeroing all
 *                            of it again is also fine; after HSS_ERR_DEVICE_TIMEOUT, do).
 *                            Two calls that share a workspace must not run at the same time
 *                            on the GPU.
 * Errors as in the four calls above; HSS_ERR_WORKSPACE_TOO_SMALL if the workspace is short.
 */
size_t hss_layer_step_workspace_bytes(int32_t num_seqs);

hss_status hss_layer_step(const hss_dims* dims, const uint16_t* P, const uint16_t* K_new,
                          const int32_t* new_ids, int64_t num_new, const uint16_t* Q,
                          int32_t rows_per_seq, uint16_t* Qp, uint16_t* A_g, int32_t layer,
                          const int32_t* block_table, const int32_t* seq_offsets,
                          int32_t num_seqs, int64_t total_blocks, float* scores, int32_t k,
                          int32_t* victims, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream);

/*
 * hss_layer_step with the arguments that stay the same from call to call bound once in a
 * struct (a serving loop's layer calls differ only in the layer, the new key blocks, the
 * queries, the outputs and the stream): one call is exactly
 *   hss_layer_step(&args->dims, args->P, K_new, args->new_ids, args->num_new, Q,
 *                  args->rows_per_seq, args->Qp, args->A_g, layer, args->block_table,
 *                  args->seq_offsets, args->num_seqs, args->total_blocks, scores, args->k,
 *                  victims, args->workspace, args->workspace_bytes, args->dev_status, stream)
 * with every argument's meaning, layout, ownership and error as there; the struct is read
 * during the call only (the caller keeps it).  A calling convention of this library (the
 * pages have no counterpart): fewer arguments to marshal per call for bindings whose
 * per-argument cost shows beside a 10 us layer call.  HSS_ERR_NULL_POINTER if args is NULL.
 */
typedef struct hss_layer_step_args {
    hss_dims dims;
    const uint16_t* P;
    const int32_t* new_ids;
    int64_t num_new;
    int32_t rows_per_seq;
    uint16_t* Qp;
    uint16_t* A_g;
    const int32_t* block_table;
    const int32_t* seq_offsets;
    int32_t num_seqs;
    int64_t total_blocks;
    int32_t k;
    void* workspace;
    size_t workspace_bytes;
    int32_t* dev_status;
} hss_layer_step_args;

hss_status hss_layer_step_bound(const hss_layer_step_args* args, int32_t layer,
                                const uint16_t* K_new, const uint16_t* Q, float* scores,
                                int32_t* victims, void* stream);

/*
 * hss_layer_step for callers that cannot allocate device memory.  (The predictor pages have
 * no counterpart: this is a calling convention of this library.)
 *
 * hss_layer_step needs a caller-allocated workspace.  Some callers cannot call cudaMalloc
 * there: an engine whose memory arena owns the GPU's memory and allows no allocation after
 * start-up, a library hosted by a process that hands it no allocator, or a caller that only
 * holds raw pointers to its own buffers.  This variant takes no workspace: the completion
 * counters live in a fixed array inside the library, HSS_LAYER_STEP_STATIC_MAX_SEQS int32
 * words and 32.25 KiB more (48.25 KiB) on every GPU that loads it, kept until the process
 * exits.  It allocates
 * nothing and calls no allocating routine.
 *
 *   Arguments and results: as hss_layer_step, without workspace / workspace_bytes; Qp must
 *   not be NULL here (HSS_ERR_NULL_POINTER).
 *   Every argument check runs before anything is enqueued, as for the other calls.
 *   num_seqs > HSS_LAYER_STEP_STATIC_MAX_SEQS  -> HSS_ERR_WORKSPACE_TOO_SMALL, nothing enqueued.
 *   Each call first clears the counters it uses (a memset on `stream`), then runs the same
 *   kernels as hss_layer_step.
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress);
 *   make that first call before any stream capture on that device.  The address is kept
 *   for the life of the process: after cudaDeviceReset on that device, reload the library
 *   before calling this again (the same holds for the library's error word).
 *   All calls share the one array: calls that overlap on the GPU (on different streams, or
 *   unordered) race and give wrong victims.  Order them on one stream.
 */
#define HSS_LAYER_STEP_STATIC_MAX_SEQS 4096

int32_t hss_layer_step_static_max_seqs(void);

hss_status hss_layer_step_static(const hss_dims* dims, const uint16_t* P, const uint16_t* K_new,
                                 const int32_t* new_ids, int64_t num_new, const uint16_t* Q,
                                 int32_t rows_per_seq, uint16_t* Qp, uint16_t* A_g, int32_t layer,
                                 const int32_t* block_table, const int32_t* seq_offsets,
                                 int32_t num_seqs, int64_t total_blocks, float* scores, int32_t k,
                                 int32_t* victims, int32_t* dev_status, void* stream);

/*
 * Failure-detection self-test.  Every pipeline wait in the tensor-core kernels gives up
 * after a time limit and reports HSS_ERR_DEVICE_TIMEOUT instead of hanging the GPU.  This
 * call launches one small kernel whose thread waits, with that same bounded wait, on a
 * barrier nothing arrives on, for limit_ns (1e3 .. 2e9) nanoseconds; the kernel then stores
 * HSS_ERR_DEVICE_TIMEOUT into *dev_status (device int32, which the caller zeroes first) and
 * into the library's error word, and exits.  The context stays usable.
 */
hss_status hss_self_test_wait_timeout(int32_t* dev_status, int64_t limit_ns, void* stream);

/*
 * Failure-detection self-test of hss_layer_step's one-sequence victim ranking.  In that
 * ranking every CTA of the scorer waits until all of the sequence's keys are published, with
 * a bounded wait.  This call runs the decode layer call's scorer on one sequence (one query
 * row, queries projected in the scorer, no new blocks; the arguments as in hss_layer_step)
 * with its last CTA withholding its keys, so that every CTA's wait runs out after limit_ns
 * (1e3 .. 2e9) nanoseconds: HSS_ERR_DEVICE_TIMEOUT is stored into *dev_status and the
 * library's error word, the kernel exits, the context stays usable.  The scores are
 * written; the victims are not meaningful.  Zero the workspace again before the next
 * hss_layer_step on it.  HSS_ERR_UNSUPPORTED_SHAPE (nothing launched) when the shape does not
 * take that ranking (more than 4096 entries, or a grid that does not fit the GPU at once).
 * No page has a counterpart: it tests this library's own wait.
 */
hss_status hss_self_test_spread_wait(const hss_dims* dims, const uint16_t* P, const uint16_t* Q,
                                     uint16_t* A_g, int32_t layer, const int32_t* block_table,
                                     const int32_t* seq_offsets, int64_t total_blocks,
                                     float* scores, int32_t k, int32_t* victims, void* workspace,
                                     size_t workspace_bytes, int64_t limit_ns,
                                     int32_t* dev_status, void* stream);

/*
 * Device-side error word of the current device: the first HSS_ERR_* code a
 * kernel raised since the last read (HSS_ERR_DEVICE_TIMEOUT when a pipeline
 * wait ran out), or HSS_OK.  Synchronises `stream`, copies the word to
 * *status and clears it.
 */
hss_status hss_read_device_error(int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* HSS_H */
