// hss_api.cu -- the C ABI (include/hss.h): host-side validation, per-device set-up and
// dispatch to the kernels.  Every check runs before anything is enqueued, so a call that
// returns an error has launched nothing.
#include <mutex>

#include "internal.h"

namespace hss {
namespace {

// The library's own device error word (one per device that loads the library).
__device__ int32_t g_device_error = 0;

constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_info_ready[kMaxDevices] = {false};
std::mutex g_info_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

const DeviceInfo* current_device_info() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_info_mu);
    if (!g_info_ready[dev]) {
        DeviceInfo info;
        info.device = dev;
        if (cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                   dev) != cudaSuccess) {
            return nullptr;
        }
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return nullptr;
        info.error_word = static_cast<int32_t*>(addr);
        g_info[dev] = info;
        g_info_ready[dev] = true;
    }
    return &g_info[dev];
}

static hss_status check_dims(const hss_dims* d) {
    if (d == nullptr) return HSS_ERR_NULL_POINTER;
    if (d->num_layers <= 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 ||
        d->r <= 0 || d->block_size <= 0 || d->max_blocks <= 0)
        return HSS_ERR_INVALID_DIMS;
    if (d->num_q_heads % d->num_kv_heads != 0) return HSS_ERR_INVALID_DIMS;
    if (d->max_blocks > 0x7FFFFFFF) return HSS_ERR_UNSUPPORTED_SHAPE;
    if (d->num_kv_heads > 64) return HSS_ERR_UNSUPPORTED_SHAPE;
    if (d->r != 16 && d->r != 32 && d->r != 64 && d->r != 128) return HSS_ERR_UNSUPPORTED_SHAPE;
    if (d->block_size % 16 != 0 || d->block_size > 256) return HSS_ERR_UNSUPPORTED_SHAPE;
    if (d->head_dim % 64 != 0 || d->head_dim > 256) return HSS_ERR_UNSUPPORTED_SHAPE;
    return HSS_OK;
}


hss_status layer_step_check(const hss_dims* dims, const uint16_t* P, const uint16_t* K_new,
                            const int32_t* new_ids, int64_t num_new, const uint16_t* Q,
                            int32_t rows_per_seq, const uint16_t* Qp, const uint16_t* A_g,
                            int32_t layer, const int32_t* block_table,
                            const int32_t* seq_offsets, int32_t num_seqs, int64_t total_blocks,
                            const float* scores, int32_t k, const int32_t* victims,
                            const void* workspace, size_t workspace_bytes, LayerStepPlan* plan) {
    hss_status st = check_dims(dims);
    if (st != HSS_OK) return st;
    if (layer < 0 || layer >= dims->num_layers) return HSS_ERR_OUT_OF_RANGE;
    if (num_new < 0 || num_seqs < 0 || total_blocks < 0 || rows_per_seq < 1 ||
        total_blocks > 0x7FFFFFFF || k < 1 || k > HSS_MAX_VICTIMS)
        return HSS_ERR_INVALID_ARGUMENT;
    if (num_seqs == 0 && total_blocks != 0) return HSS_ERR_INVALID_ARGUMENT;
    if (P == nullptr || A_g == nullptr) return HSS_ERR_NULL_POINTER;
    if (num_new > 0 && (K_new == nullptr || new_ids == nullptr)) return HSS_ERR_NULL_POINTER;
    if (num_seqs > 0 && (Q == nullptr || seq_offsets == nullptr || victims == nullptr))
        return HSS_ERR_NULL_POINTER;
    if (total_blocks > 0 && (block_table == nullptr || scores == nullptr))
        return HSS_ERR_NULL_POINTER;
    if (!aligned16(P) || !aligned16(A_g) || (K_new != nullptr && !aligned16(K_new)) ||
        (Q != nullptr && !aligned16(Q)) || (Qp != nullptr && !aligned16(Qp)))
        return HSS_ERR_MISALIGNED;
    if (num_seqs > 0) {
        if (workspace == nullptr) return HSS_ERR_NULL_POINTER;
        if (workspace_bytes < hss_layer_step_workspace_bytes(num_seqs))
            return HSS_ERR_WORKSPACE_TOO_SMALL;
        if ((reinterpret_cast<uintptr_t>(workspace) & 3u) != 0) return HSS_ERR_MISALIGNED;
    }
    const int64_t rows_per_block = static_cast<int64_t>(dims->block_size) * dims->num_kv_heads;
    if (num_new > (int64_t{1} << 31) / rows_per_block) return HSS_ERR_INVALID_ARGUMENT;
    if (static_cast<int64_t>(num_seqs) * rows_per_seq > (int64_t{1} << 40) / dims->num_q_heads)
        return HSS_ERR_INVALID_ARGUMENT;

    // The scoring path, decided before anything is launched so that an unsupported shape
    // enqueues nothing.
    ScoreArgs& a = plan->score;
    a = ScoreArgs{};
    a.Qp = Qp;
    a.rows_per_seq = rows_per_seq;
    a.A_g = A_g;
    a.layer_offset_slots = static_cast<int64_t>(layer) * dims->max_blocks;
    a.max_blocks = dims->max_blocks;
    a.table = block_table;
    a.seq_offsets = seq_offsets;
    a.num_seqs = num_seqs;
    a.total = total_blocks;
    a.scores = const_cast<float*>(scores);
    a.num_q_heads = dims->num_q_heads;
    a.num_kv_heads = dims->num_kv_heads;
    a.r = dims->r;
    a.block_size = dims->block_size;
    const int64_t nvec =
        static_cast<int64_t>(rows_per_seq) * (dims->num_q_heads / dims->num_kv_heads);
    plan->decode = nvec <= 16 && score_decode_supported(a);
    if (total_blocks > 0 && !plan->decode && !score_tc_supported(a))
        return HSS_ERR_UNSUPPORTED_SHAPE;
    // Qp == NULL: the caller does not want the projected queries, and the decode scorer
    // projects them itself (one launch fewer on the scoring path).
    plan->inline_q = Qp == nullptr && num_seqs > 0;
    if (plan->inline_q && total_blocks > 0 &&
        !(plan->decode && score_decode_inline_supported(a, dims->head_dim)))
        return HSS_ERR_NULL_POINTER;
    return HSS_OK;
}

}  // namespace hss

using namespace hss;

extern "C" {

const char* hss_status_string(int32_t status) {
    switch (status) {
        case HSS_OK: return "HSS_OK";
        case HSS_ERR_INVALID_DIMS: return "HSS_ERR_INVALID_DIMS";
        case HSS_ERR_OUT_OF_RANGE: return "HSS_ERR_OUT_OF_RANGE";
        case HSS_ERR_NULL_POINTER: return "HSS_ERR_NULL_POINTER";
        case HSS_ERR_MISALIGNED: return "HSS_ERR_MISALIGNED";
        case HSS_ERR_WORKSPACE_TOO_SMALL: return "HSS_ERR_WORKSPACE_TOO_SMALL";
        case HSS_ERR_UNSUPPORTED_SHAPE: return "HSS_ERR_UNSUPPORTED_SHAPE";
        case HSS_ERR_CUDA: return "HSS_ERR_CUDA";
        case HSS_ERR_DEVICE_TIMEOUT: return "HSS_ERR_DEVICE_TIMEOUT";
        case HSS_ERR_INVALID_ARGUMENT: return "HSS_ERR_INVALID_ARGUMENT";
        default: return "HSS_ERR_UNKNOWN";
    }
}

int32_t hss_version(void) { return 100; }

hss_status hss_validate_dims(const hss_dims* dims) { return check_dims(dims); }

size_t hss_a_g_bytes(const hss_dims* d) {
    if (d == nullptr || d->num_layers <= 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 ||
        d->head_dim <= 0 || d->r <= 0 || d->block_size <= 0 || d->max_blocks <= 0 ||
        d->num_q_heads % d->num_kv_heads != 0)
        return 0;
    return static_cast<size_t>(d->num_layers) * static_cast<size_t>(d->max_blocks) *
           static_cast<size_t>(d->num_kv_heads) * static_cast<size_t>(d->block_size) *
           static_cast<size_t>(d->r) * 2u;
}

hss_status hss_project_q(const hss_dims* dims, const uint16_t* P, const uint16_t* Q,
                         int64_t num_rows, uint16_t* Qp, void* stream) {
    hss_status st = check_dims(dims);
    if (st != HSS_OK) return st;
    if (num_rows < 0) return HSS_ERR_INVALID_ARGUMENT;
    if (num_rows == 0) return HSS_OK;
    if (P == nullptr || Q == nullptr || Qp == nullptr) return HSS_ERR_NULL_POINTER;
    if (!aligned16(P) || !aligned16(Q) || !aligned16(Qp)) return HSS_ERR_MISALIGNED;
    if (num_rows > (int64_t{1} << 40) / dims->num_q_heads) return HSS_ERR_INVALID_ARGUMENT;
    ProjectArgs a{};
    a.P = P;
    a.X = Q;
    a.num_rows = num_rows * dims->num_q_heads;
    a.head_dim = dims->head_dim;
    a.r = dims->r;
    a.out = Qp;
    a.block_ids = nullptr;
    return launch_project(a, static_cast<cudaStream_t>(stream));
}

hss_status hss_project_kv_blocks(const hss_dims* dims, const uint16_t* P, const uint16_t* K,
                                 int32_t layer, const int32_t* block_ids, int64_t num_blocks,
                                 uint16_t* A_g, int32_t* dev_status, void* stream) {
    hss_status st = check_dims(dims);
    if (st != HSS_OK) return st;
    if (layer < 0 || layer >= dims->num_layers) return HSS_ERR_OUT_OF_RANGE;
    if (num_blocks < 0) return HSS_ERR_INVALID_ARGUMENT;
    if (num_blocks == 0) return HSS_OK;
    if (P == nullptr || K == nullptr || block_ids == nullptr || A_g == nullptr)
        return HSS_ERR_NULL_POINTER;
    if (!aligned16(P) || !aligned16(K) || !aligned16(A_g)) return HSS_ERR_MISALIGNED;
    const int64_t rows_per_block = static_cast<int64_t>(dims->block_size) * dims->num_kv_heads;
    if (num_blocks > (int64_t{1} << 31) / rows_per_block) return HSS_ERR_INVALID_ARGUMENT;
    ProjectArgs a{};
    a.P = P;
    a.X = K;
    a.num_rows = num_blocks * rows_per_block;
    a.head_dim = dims->head_dim;
    a.r = dims->r;
    a.out = A_g;
    a.block_ids = block_ids;
    a.num_kv_heads = dims->num_kv_heads;
    a.block_size = dims->block_size;
    a.max_blocks = dims->max_blocks;
    a.layer = layer;
    a.dev_status = dev_status;
    return launch_project(a, static_cast<cudaStream_t>(stream));
}

hss_status hss_write_kv_tokens(const hss_dims* dims, const uint16_t* P, const uint16_t* K_tok,
                               const int64_t* slots, int64_t num_tokens, uint16_t* K_cache,
                               uint16_t* A_g, int32_t layer, int32_t* dev_status, void* stream) {
    hss_status st = check_dims(dims);
    if (st != HSS_OK) return st;
    if (layer < 0 || layer >= dims->num_layers) return HSS_ERR_OUT_OF_RANGE;
    if (num_tokens < 0) return HSS_ERR_INVALID_ARGUMENT;
    if (num_tokens == 0) return HSS_OK;
    if (P == nullptr || K_tok == nullptr || slots == nullptr || A_g == nullptr)
        return HSS_ERR_NULL_POINTER;
    if (!aligned16(P) || !aligned16(K_tok) || !aligned16(A_g) ||
        (K_cache != nullptr && !aligned16(K_cache)) || (reinterpret_cast<uintptr_t>(slots) & 7u))
        return HSS_ERR_MISALIGNED;
    if (num_tokens > (int64_t{1} << 31) / dims->num_kv_heads) return HSS_ERR_INVALID_ARGUMENT;
    ProjectArgs a{};
    a.P = P;
    a.X = K_tok;
    a.num_rows = num_tokens * dims->num_kv_heads;
    a.head_dim = dims->head_dim;
    a.r = dims->r;
    a.out = A_g;
    a.slots = slots;
    a.cache = K_cache;
    a.num_kv_heads = dims->num_kv_heads;
    a.block_size = dims->block_size;
    a.max_blocks = dims->max_blocks;
    a.layer = layer;
    a.dev_status = dev_status;
    return launch_project(a, static_cast<cudaStream_t>(stream));
}

hss_status hss_score_blocks(const hss_dims* dims, const uint16_t* Qp, int32_t rows_per_seq,
                            const uint16_t* A_g, int32_t layer, const int32_t* block_table,
                            const int32_t* seq_offsets, int32_t num_seqs, int64_t total_blocks,
                            float* scores, int32_t path, int32_t* dev_status, void* stream) {
    return hss_score_blocks_masked(dims, Qp, rows_per_seq, A_g, layer, block_table, seq_offsets,
                                   num_seqs, total_blocks, nullptr, nullptr, scores, path,
                                   dev_status, stream);
}

hss_status hss_score_blocks_masked(const hss_dims* dims, const uint16_t* Qp, int32_t rows_per_seq,
                                   const uint16_t* A_g, int32_t layer, const int32_t* block_table,
                                   const int32_t* seq_offsets, int32_t num_seqs,
                                   int64_t total_blocks, const int32_t* ctx_len,
                                   const int32_t* row_pos0, float* scores, int32_t path,
                                   int32_t* dev_status, void* stream) {
    hss_status st = check_dims(dims);
    if (st != HSS_OK) return st;
    if (layer < 0 || layer >= dims->num_layers) return HSS_ERR_OUT_OF_RANGE;
    if (num_seqs < 0 || total_blocks < 0 || rows_per_seq < 1 || total_blocks > 0x7FFFFFFF)
        return HSS_ERR_INVALID_ARGUMENT;
    if (path != HSS_PATH_AUTO && path != HSS_PATH_DECODE && path != HSS_PATH_TCGEN05)
        return HSS_ERR_INVALID_ARGUMENT;
    if (num_seqs == 0 && total_blocks != 0) return HSS_ERR_INVALID_ARGUMENT;
    if (total_blocks == 0) return HSS_OK;
    if (Qp == nullptr || A_g == nullptr || block_table == nullptr || seq_offsets == nullptr ||
        scores == nullptr)
        return HSS_ERR_NULL_POINTER;
    if (!aligned16(Qp) || !aligned16(A_g)) return HSS_ERR_MISALIGNED;
    ScoreArgs a{};
    a.Qp = Qp;
    a.rows_per_seq = rows_per_seq;
    a.A_g = A_g;
    a.layer_offset_slots = static_cast<int64_t>(layer) * dims->max_blocks;
    a.max_blocks = dims->max_blocks;
    a.table = block_table;
    a.seq_offsets = seq_offsets;
    a.num_seqs = num_seqs;
    a.total = total_blocks;
    a.scores = scores;
    a.num_q_heads = dims->num_q_heads;
    a.num_kv_heads = dims->num_kv_heads;
    a.r = dims->r;
    a.block_size = dims->block_size;
    a.dev_status = dev_status;
    a.ctx_len = ctx_len;
    a.row_pos0 = row_pos0;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t nvec = static_cast<int64_t>(rows_per_seq) * (dims->num_q_heads / dims->num_kv_heads);
    int chosen = path;
    if (chosen == HSS_PATH_AUTO) {
        chosen = (nvec <= 16 && score_decode_supported(a)) ? HSS_PATH_DECODE : HSS_PATH_TCGEN05;
    }
    if (chosen == HSS_PATH_DECODE) {
        if (!score_decode_supported(a)) return HSS_ERR_UNSUPPORTED_SHAPE;
        return launch_score_decode(a, s);
    }
    if (!score_tc_supported(a)) return HSS_ERR_UNSUPPORTED_SHAPE;
    return launch_score_tc(a, s);
}

hss_status hss_rank_victims(const float* scores, const int32_t* seq_offsets, int32_t num_seqs,
                            int64_t total_blocks, int32_t k, int32_t* victims, void* stream) {
    if (num_seqs < 0 || total_blocks < 0 || total_blocks > 0x7FFFFFFF)
        return HSS_ERR_INVALID_ARGUMENT;
    if (k < 1 || k > HSS_MAX_VICTIMS) return HSS_ERR_INVALID_ARGUMENT;
    if (num_seqs == 0) return HSS_OK;
    if (seq_offsets == nullptr || victims == nullptr || (scores == nullptr && total_blocks > 0))
        return HSS_ERR_NULL_POINTER;
    return launch_rank_victims(scores, seq_offsets, num_seqs, total_blocks, k, victims,
                               static_cast<cudaStream_t>(stream));
}

size_t hss_layer_step_workspace_bytes(int32_t num_seqs) {
    if (num_seqs <= 0) return 0;
    // The one-sequence spread ranking's region (its call number in 256 bytes, then 8 bytes for
    // each of at most 4096 entries), then the per-sequence completion counters (rounded up to
    // 256 bytes).
    const size_t b = static_cast<size_t>(num_seqs) * sizeof(int32_t);
    return static_cast<size_t>(kSpreadRegionBytes) + (b + 255) / 256 * 256;
}

hss_status hss_layer_step(const hss_dims* dims, const uint16_t* P, const uint16_t* K_new,
                          const int32_t* new_ids, int64_t num_new, const uint16_t* Q,
                          int32_t rows_per_seq, uint16_t* Qp, uint16_t* A_g, int32_t layer,
                          const int32_t* block_table, const int32_t* seq_offsets,
                          int32_t num_seqs, int64_t total_blocks, float* scores, int32_t k,
                          int32_t* victims, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream) {
    LayerStepPlan plan;
    hss_status st = layer_step_check(dims, P, K_new, new_ids, num_new, Q, rows_per_seq, Qp, A_g,
                                     layer, block_table, seq_offsets, num_seqs, total_blocks,
                                     scores, k, victims, workspace, workspace_bytes, &plan);
    if (st != HSS_OK) return st;
    const ScoreArgs& a = plan.score;
    const int64_t rows_per_block = static_cast<int64_t>(dims->block_size) * dims->num_kv_heads;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // 1. one launch projects the query rows and the newly written blocks
    {
        ProjectArgs q{};
        q.P = P;
        q.X = Q;
        q.num_rows = plan.inline_q ? 0 : static_cast<int64_t>(num_seqs) * rows_per_seq *
                                             dims->num_q_heads;
        q.head_dim = dims->head_dim;
        q.r = dims->r;
        q.out = Qp;
        q.block_ids = nullptr;
        ProjectArgs kv{};
        kv.P = P;
        kv.X = K_new;
        kv.num_rows = num_new * rows_per_block;
        kv.head_dim = dims->head_dim;
        kv.r = dims->r;
        kv.out = A_g;
        kv.block_ids = new_ids;
        kv.num_kv_heads = dims->num_kv_heads;
        kv.block_size = dims->block_size;
        kv.max_blocks = dims->max_blocks;
        kv.layer = layer;
        kv.dev_status = dev_status;
        st = launch_project2(q, &kv, s);
        if (st != HSS_OK || num_seqs == 0) return st;
    }
    // 2. scores, with the ranking fused into the decode scorer where it fits
    bool fused = false;
    if (total_blocks > 0) {
        ScoreArgs sa = a;
        sa.dev_status = dev_status;
        if (plan.decode) {
            // The kernel just before the scorer is this call's projection unless the queries
            // are projected in the scorer and there are no new blocks: then nothing of this
            // call precedes it and it may read nothing before its dependency wait.
            const bool own_projection = !plan.inline_q || num_new > 0;
            int32_t* ws = static_cast<int32_t*>(workspace);
            const FusedRank fr{ws + kSpreadRegionBytes / 4, ws, victims, k, own_projection,
                               new_ids, num_new};
            // With the queries projected in the scorer, that projection writes only the new
            // slots, so the scorer need not wait for it anywhere else.
            const InlineQ iq{Q, P, dims->head_dim, num_new > 0};
            st = launch_score_decode(sa, s, &fr, &fused, plan.inline_q ? &iq : nullptr);
        } else {
            st = launch_score_tc(sa, s);
        }
        if (st != HSS_OK) return st;
    }
    // 3. otherwise a separate ranking launch
    if (!fused) return launch_rank_victims(scores, seq_offsets, num_seqs, total_blocks, k, victims, s);
    return HSS_OK;
}

hss_status hss_layer_step_bound(const hss_layer_step_args* args, int32_t layer,
                                const uint16_t* K_new, const uint16_t* Q, float* scores,
                                int32_t* victims, void* stream) {
    if (args == nullptr) return HSS_ERR_NULL_POINTER;
    return hss_layer_step(&args->dims, args->P, K_new, args->new_ids, args->num_new, Q,
                          args->rows_per_seq, args->Qp, args->A_g, layer, args->block_table,
                          args->seq_offsets, args->num_seqs, args->total_blocks, scores, args->k,
                          victims, args->workspace, args->workspace_bytes, args->dev_status,
                          stream);
}

hss_status hss_self_test_spread_wait(const hss_dims* dims, const uint16_t* P, const uint16_t* Q,
                                     uint16_t* A_g, int32_t layer, const int32_t* block_table,
                                     const int32_t* seq_offsets, int64_t total_blocks,
                                     float* scores, int32_t k, int32_t* victims, void* workspace,
                                     size_t workspace_bytes, int64_t limit_ns,
                                     int32_t* dev_status, void* stream) {
    if (limit_ns < 1000 || limit_ns > 2000000000) return HSS_ERR_INVALID_ARGUMENT;
    LayerStepPlan plan;
    hss_status st = layer_step_check(dims, P, nullptr, nullptr, 0, Q, 1, nullptr, A_g, layer,
                                     block_table, seq_offsets, 1, total_blocks, scores, k,
                                     victims, workspace, workspace_bytes, &plan);
    if (st != HSS_OK) return st;
    if (total_blocks == 0 || !plan.decode || !plan.inline_q) return HSS_ERR_UNSUPPORTED_SHAPE;
    int32_t* ws = static_cast<int32_t*>(workspace);
    FusedRank fr{ws + kSpreadRegionBytes / 4, ws, victims, k, false, nullptr, 0};
    fr.wait_limit_ns = limit_ns;
    fr.withhold_cta = 0x7FFFFFFF;  // past the grid: its last CTA
    fr.require_spread = true;
    ScoreArgs sa = plan.score;
    sa.dev_status = dev_status;
    const InlineQ iq{Q, P, dims->head_dim, false};
    bool fused = false;
    return launch_score_decode(sa, static_cast<cudaStream_t>(stream), &fr, &fused, &iq);
}

hss_status hss_score_rows(const hss_dims* dims, const uint16_t* Qp, int32_t rows,
                          const uint16_t* A_g, int32_t layer, const int32_t* block_table,
                          int64_t num_blocks, float* scores, int32_t* dev_status, void* stream) {
    hss_status st = check_dims(dims);
    if (st != HSS_OK) return st;
    if (layer < 0 || layer >= dims->num_layers) return HSS_ERR_OUT_OF_RANGE;
    if (rows < 1 || num_blocks < 0 || num_blocks > 0x7FFFFFFF ||
        static_cast<int64_t>(rows) * num_blocks > (int64_t{1} << 40))
        return HSS_ERR_INVALID_ARGUMENT;
    if (num_blocks == 0) return HSS_OK;
    if (Qp == nullptr || A_g == nullptr || block_table == nullptr || scores == nullptr)
        return HSS_ERR_NULL_POINTER;
    if (!aligned16(Qp) || !aligned16(A_g) || (reinterpret_cast<uintptr_t>(scores) & 3u))
        return HSS_ERR_MISALIGNED;
    const int g = dims->num_q_heads / dims->num_kv_heads;
    ScoreArgs a{};
    a.Qp = Qp;
    a.rows_per_seq = rows;
    a.A_g = A_g;
    a.layer_offset_slots = static_cast<int64_t>(layer) * dims->max_blocks;
    a.max_blocks = dims->max_blocks;
    a.table = block_table;
    a.seq_offsets = nullptr;
    a.num_seqs = 1;
    a.total = num_blocks;
    a.scores = scores;
    a.num_q_heads = dims->num_q_heads;
    a.num_kv_heads = dims->num_kv_heads;
    a.r = dims->r;
    a.block_size = dims->block_size;
    a.dev_status = dev_status;
    if ((g & (g - 1)) != 0 || g > 16 || !score_tc_supported(a)) return HSS_ERR_UNSUPPORTED_SHAPE;
    return launch_score_tc_rows(a, static_cast<cudaStream_t>(stream));
}

hss_status hss_select_rows(const float* scores, int32_t rows, int64_t num_blocks,
                           int64_t first_pos, int32_t block_size, int32_t topk, int32_t* lists,
                           void* stream) {
    if (rows < 0 || num_blocks < 0 || num_blocks > 0x7FFFFFFF || first_pos < 0 ||
        block_size < 1 || topk < 1 || topk > HSS_MAX_VICTIMS)
        return HSS_ERR_INVALID_ARGUMENT;
    if (rows == 0) return HSS_OK;
    if (lists == nullptr || (num_blocks > 0 && scores == nullptr)) return HSS_ERR_NULL_POINTER;
    if ((reinterpret_cast<uintptr_t>(scores) & 3u) || (reinterpret_cast<uintptr_t>(lists) & 3u))
        return HSS_ERR_MISALIGNED;
    return launch_select_rows(scores, rows, num_blocks, first_pos, block_size, topk, lists,
                              static_cast<cudaStream_t>(stream));
}

hss_status hss_read_device_error(int32_t* status, void* stream) {
    if (status == nullptr) return HSS_ERR_NULL_POINTER;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (current_device_info() == nullptr) return HSS_ERR_CUDA;
    int32_t v = 0;
    const int32_t zero = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return HSS_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return HSS_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return HSS_ERR_CUDA;
    *status = v;
    return HSS_OK;
}

}  // extern "C"
