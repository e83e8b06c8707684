// rank.cu -- eviction victims: per sequence, the k table entries with the smallest scores.
//
// The predictor page ("metrale_storage/predictor.rs", module docs) uses block scores only to
// rank eviction victims; the order of equal scores (lower index first) mirrors the host top-k
// of "metrale_model_layers/layers/qsa_select.rs".  Each score becomes an order-preserving
// 32-bit key (-0 -> +0, NaN -> +inf); the words (key << 32 | index) are then unique, so the
// answer is exact and unambiguous.
//
// One CTA per sequence: 256 threads when the average sequence is at most 4096 entries
// (its keys then sit in registers, 16 per thread), 1024 otherwise (8 per thread).  The selection itself is
// rank_sequence in rank_device.cuh, shared with the fused decode scorer.
#include <algorithm>

#include "rank_device.cuh"

namespace hss {
namespace {

using rankdev::RankShared;

template <int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
    rank_kernel(const float* __restrict__ scores, const int32_t* __restrict__ seq_offsets, int k,
                int sel_cap, int32_t* __restrict__ victims) {
    extern __shared__ uint8_t smem_raw[];
    uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw);  // [sel_cap]
    RankShared* sh = reinterpret_cast<RankShared*>(sel + sel_cap);
    grid_dependency_wait();
    grid_launch_dependents();
    const int s = blockIdx.x;
    const int64_t base = seq_offsets[s];
    const int n = static_cast<int>(seq_offsets[s + 1] - base);
    rankdev::rank_sequence<THREADS>(scores + base, n, k, victims + static_cast<int64_t>(s) * k,
                                    sel, sel_cap, sh);
}

// One CTA per query row: the row's complete blocks, largest score first.
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
    select_rows_kernel(const float* __restrict__ scores, int64_t n, int64_t first_pos,
                       int block_size, int topk, int sel_cap, int32_t* __restrict__ lists) {
    extern __shared__ uint8_t smem_raw[];
    uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw);  // [sel_cap]
    RankShared* sh = reinterpret_cast<RankShared*>(sel + sel_cap);
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t row = blockIdx.x;
    int64_t complete = (first_pos + row + 1) / block_size;
    complete = complete < 0 ? 0 : (complete > n ? n : complete);
    rankdev::rank_sequence<THREADS, true>(scores + row * n, static_cast<int>(complete), topk,
                                          lists + row * topk, sel, sel_cap, sh);
}

int g_set_small[64] = {0};
int g_set_rows_small[64] = {0};
int g_set_rows_large[64] = {0};
int g_set_large[64] = {0};

}  // namespace

hss_status launch_rank_victims(const float* scores, const int32_t* seq_offsets, int32_t num_seqs,
                               int64_t total, int32_t k, int32_t* victims, cudaStream_t stream) {
    if (num_seqs == 0) return HSS_OK;
    const DeviceInfo* dev = current_device_info();
    if (dev == nullptr) return HSS_ERR_CUDA;
    const int sel_cap = rankdev::rank_sel_cap(k);
    const int smem = rankdev::rank_smem_bytes(sel_cap);
    const bool small = total / num_seqs <= 4096;
    auto kern = small ? rank_kernel<256> : rank_kernel<1024>;
    int* set = small ? g_set_small : g_set_large;
    const int d = dev->device & 63;
    if (set[d] < smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return HSS_ERR_CUDA;
        set[d] = smem;
    }
    if (launch_pdl(kern, dim3(num_seqs), dim3(small ? 256 : 1024), smem, stream, scores,
                   seq_offsets, k, sel_cap, victims) != cudaSuccess)
        return HSS_ERR_CUDA;
    return HSS_OK;
}

hss_status launch_select_rows(const float* scores, int32_t rows, int64_t n, int64_t first_pos,
                              int32_t block_size, int32_t topk, int32_t* lists,
                              cudaStream_t stream) {
    if (rows == 0) return HSS_OK;
    const DeviceInfo* dev = current_device_info();
    if (dev == nullptr) return HSS_ERR_CUDA;
    const int sel_cap = rankdev::rank_sel_cap(topk);
    const int smem = rankdev::rank_smem_bytes(sel_cap);
    const bool small = n <= 4096;
    auto kern = small ? select_rows_kernel<256> : select_rows_kernel<1024>;
    int* set = small ? g_set_rows_small : g_set_rows_large;
    const int d = dev->device & 63;
    if (set[d] < smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return HSS_ERR_CUDA;
        set[d] = smem;
    }
    if (launch_pdl(kern, dim3(rows), dim3(small ? 256 : 1024), smem, stream, scores, n,
                   first_pos, static_cast<int>(block_size), static_cast<int>(topk), sel_cap,
                   lists) != cudaSuccess)
        return HSS_ERR_CUDA;
    return HSS_OK;
}

}  // namespace hss
