// rank.cu -- eviction victims: per sequence, the k table entries with the smallest scores.
//
// The predictor page ("metrale_storage/predictor.rs", module docs) uses block scores only to
// rank eviction victims; the order of equal scores (lower index first) mirrors the host top-k
// of "metrale_model_layers/layers/qsa_select.rs".  Each score becomes an order-preserving
// 32-bit key (-0 -> +0, NaN -> +inf); the words (key << 32 | index) are then unique, so the
// answer is exact and unambiguous.
//
// One CTA per sequence (256 threads for short sequences, 1024 for long ones):
//   1. radix select, four 8-bit digits from the top (double-buffered histograms, two
//      barriers per digit), finds the key T of the k-th smallest entry, how many keys equal
//      T are still needed, and how many keys equal T there are;
//   2. if every key <= T fits in the selection buffer (the usual case), one pass appends them
//      all (warp-aggregated atomics) and the sort below orders ties by index for free;
//      otherwise (a mass of ties at T) an ordered pass appends the keys < T and the first
//      `need` keys == T in index order (block-wide ballot scan);
//   3. a bitonic sort of the selected words: stages whose partner is in another warp go
//      through shared memory, stages within a warp run in registers with shuffles.
// Keys stay in shared memory when the sequence fits (<= 16384 entries); longer sequences
// re-read the (L2-resident) scores on each pass.
#include <algorithm>

#include "rank_device.cuh"

namespace hss {
namespace {

using rankdev::kKeysCap;
using rankdev::RankShared;

template <int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
    rank_kernel(const float* __restrict__ scores, const int32_t* __restrict__ seq_offsets, int k,
                int sel_cap, int keys_cap, int32_t* __restrict__ victims) {
    extern __shared__ uint8_t smem_raw[];
    uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw);  // [sel_cap]
    RankShared* sh = reinterpret_cast<RankShared*>(sel + sel_cap);
    uint32_t* keys = reinterpret_cast<uint32_t*>(sh + 1);   // [keys_cap]
    grid_dependency_wait();
    grid_launch_dependents();
    const int s = blockIdx.x;
    const int64_t base = seq_offsets[s];
    const int n = static_cast<int>(seq_offsets[s + 1] - base);
    rankdev::rank_sequence<THREADS>(scores + base, n, k, victims + static_cast<int64_t>(s) * k,
                                    sel, sel_cap, sh, keys, keys_cap);
}

int g_set_small[64] = {0};
int g_set_large[64] = {0};

}  // namespace

hss_status launch_rank_victims(const float* scores, const int32_t* seq_offsets, int32_t num_seqs,
                               int64_t total, int32_t k, int32_t* victims, cudaStream_t stream) {
    if (num_seqs == 0) return HSS_OK;
    const DeviceInfo* dev = current_device_info();
    if (dev == nullptr) return HSS_ERR_CUDA;
    const int sel_cap = rankdev::rank_sel_cap(k);
    const int keys_cap =
        static_cast<int>(std::min<int64_t>(kKeysCap, std::max<int64_t>(total, 1)));
    const int smem = rankdev::rank_smem_bytes(sel_cap, keys_cap);
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
                   seq_offsets, k, sel_cap, keys_cap, victims) != cudaSuccess)
        return HSS_ERR_CUDA;
    return HSS_OK;
}

}  // namespace hss
