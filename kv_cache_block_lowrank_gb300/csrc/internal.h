// internal.h -- declarations shared by the library's translation units (host launchers and
// the constants their kernels agree on).  Not part of the public C ABI (include/hss.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/hss.h"

namespace hss {

// A pipeline wait that has not completed after this much wall time is abandoned and
// reported as HSS_ERR_DEVICE_TIMEOUT (no kernel here legitimately waits this long).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Per-device facts the launchers need, read once per device.
struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    int max_smem_optin = 0;
    int32_t* error_word = nullptr;  // library's own device error word (device address)
};

// Returns the info of the current device, initialising it on first use.  nullptr on failure.
const DeviceInfo* current_device_info();

// Launch with programmatic stream serialization: the kernel may be scheduled while the
// previous kernel in the stream finishes; it waits for it (griddepcontrol.wait) before
// touching global memory, so only launch latency and on-chip set-up overlap.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
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
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ------------------------------------------------------------------- projection (tcgen05)
// Y rows = bf16(X rows . P).  X is [num_rows, head_dim] bf16.  Output row m goes to
//   - Qp mode (block_ids == nullptr): out + m * r
//   - A_g mode: row m = (i * block_size + t) * num_kv_heads + h goes to the A_g slot row
//     ((layer * max_blocks + block_ids[i]) * num_kv_heads + h) * block_size + t.
struct ProjectArgs {
    const uint16_t* P;
    const uint16_t* X;
    int64_t num_rows;
    int32_t head_dim;
    int32_t r;
    uint16_t* out;
    // A_g modes: block_ids (whole blocks, rows in the page's k_block order) or slots (one
    // row per (token, kv head): token i goes to slot slots[i] = block * block_size + t,
    // negative = padding; cache, if not null, gets a copy of the key row at that slot)
    const int32_t* block_ids;
    const int64_t* slots;
    uint16_t* cache;
    int32_t num_kv_heads;
    int32_t block_size;
    int64_t max_blocks;
    int32_t layer;
    int32_t* dev_status;
};
hss_status launch_project(const ProjectArgs& a, cudaStream_t stream);
// Both segments in one launch (a1 may be nullptr or empty); they must share head_dim and r.
hss_status launch_project2(const ProjectArgs& a0, const ProjectArgs* a1, cudaStream_t stream);
bool project_shape_supported(int32_t head_dim, int32_t r);

// ------------------------------------------------------------------- decode scorer
struct ScoreArgs {
    const uint16_t* Qp;
    int32_t rows_per_seq;
    const uint16_t* A_g;
    int64_t layer_offset_slots;  // layer * max_blocks
    int64_t max_blocks;
    const int32_t* table;
    const int32_t* seq_offsets;
    int32_t num_seqs;
    int64_t total;
    float* scores;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t r;
    int32_t block_size;
    int32_t* dev_status;
    // Optional masks (device int32 per sequence, nullptr = off): only tokens at position
    // p < ctx_len[s] count; with row_pos0, row r only sees p <= row_pos0[s] + r.  Token t of
    // the entry at table position j of its sequence sits at p = j * block_size + t.
    const int32_t* ctx_len = nullptr;
    const int32_t* row_pos0 = nullptr;
};
// Victim ranking fused into the decode scorer: counters are the caller's per-sequence
// completion counters (zero on entry, left zero on exit).
// The layer-step workspace: first the one-sequence spread ranking's region (a call number in
// a 256-byte line of its own, then one 8-byte tagged key per entry, at most 4096), then the
// per-sequence completion counters.  The region comes first so that calls with different
// numbers of sequences find their counters and it at the same places.
constexpr int64_t kSpreadRegionBytes = 256 + 8 * 4096;

struct FusedRank {
    int32_t* counters;  // nullptr: no fused ranking
    int32_t* spread_region;  // the workspace's spread-ranking region (nullptr: none)
    int32_t* victims;
    int32_t k;
    // The kernel launched just before the scorer on this stream writes only Qp and the A_g
    // slots in new_ids (it is this call's own projection): the scorer may read the table
    // and the other slots before its grid dependency wait.
    bool early;
    const int32_t* new_ids;
    int64_t num_new;
    // Self-test of the one-sequence ranking's bounded wait: its limit (0: the library's), a CTA
    // that withholds its keys (-1: none), and whether the call must take that ranking (else
    // HSS_ERR_UNSUPPORTED_SHAPE, nothing launched).
    int64_t wait_limit_ns = 0;
    int32_t withhold_cta = -1;
    bool require_spread = false;
};
// Queries projected inside the decode scorer (a.Qp unused): Q [num_seqs, rows, nq, hd] and
// P [hd, r].  nowait: the kernel just before the scorer is this call's projection of the
// fr->new_ids slots alone (fr->num_new <= 32), so only warps reading those slots wait for it.
struct InlineQ {
    const uint16_t* Q;
    const uint16_t* P;
    int32_t head_dim;
    bool nowait;
};
// With fr != nullptr the ranking is fused when the shape allows; *fused reports whether it
// was (otherwise the caller must rank separately).  With iq != nullptr the queries are
// projected in the scorer; score_decode_inline_supported must hold.
hss_status launch_score_decode(const ScoreArgs& a, cudaStream_t stream,
                               const FusedRank* fr = nullptr, bool* fused = nullptr,
                               const InlineQ* iq = nullptr);
bool score_decode_supported(const ScoreArgs& a);
bool score_decode_inline_supported(const ScoreArgs& a, int32_t head_dim);
hss_status launch_score_tc(const ScoreArgs& a, cudaStream_t stream);
// Per-row scores of one sequence (a.num_seqs == 1, g = num_q_heads / num_kv_heads in
// {1, 2, 4, 8, 16}, no masks): a.scores is [rows_per_seq, total]; a.seq_offsets may be null.
hss_status launch_score_tc_rows(const ScoreArgs& a, cudaStream_t stream);
bool score_tc_supported(const ScoreArgs& a);

// ------------------------------------------------------------------- victims
// Per-row selection: row r of scores [rows, n] takes its topk largest among the first
// min(n, (first_pos + r + 1) / block_size) entries (lower index first on ties).
hss_status launch_select_rows(const float* scores, int32_t rows, int64_t n, int64_t first_pos,
                              int32_t block_size, int32_t topk, int32_t* lists,
                              cudaStream_t stream);
hss_status launch_rank_victims(const float* scores, const int32_t* seq_offsets, int32_t num_seqs,
                               int64_t total, int32_t k, int32_t* victims, cudaStream_t stream);

// ------------------------------------------------------------------- layer step
// Every argument check of hss_layer_step, and the path it takes, decided before anything is
// enqueued (hss_layer_step and hss_layer_step_static both run it first).
struct LayerStepPlan {
    ScoreArgs score;
    bool decode = false;    // the decode scorer (else the tcgen05 scorer)
    bool inline_q = false;  // the decode scorer projects the queries (Qp == NULL)
};
hss_status layer_step_check(const hss_dims* dims, const uint16_t* P, const uint16_t* K_new,
                            const int32_t* new_ids, int64_t num_new, const uint16_t* Q,
                            int32_t rows_per_seq, const uint16_t* Qp, const uint16_t* A_g,
                            int32_t layer, const int32_t* block_table,
                            const int32_t* seq_offsets, int32_t num_seqs, int64_t total_blocks,
                            const float* scores, int32_t k, const int32_t* victims,
                            const void* workspace, size_t workspace_bytes, LayerStepPlan* plan);

}  // namespace hss
