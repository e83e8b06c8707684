// rank.cu -- eviction victims: per sequence, the k table entries with the smallest scores.
//
// The predictor page ("metrale_storage/predictor.rs", module docs) uses block scores only to
// rank eviction victims; the order of equal scores (lower index first) mirrors the host top-k
// of "metrale_model_layers/layers/qsa_select.rs".  Each score becomes an order-preserving
// 32-bit key (-0 -> +0, NaN -> +inf); (key, index) pairs are then unique, so the answer is
// exact and unambiguous.
//
// One CTA per sequence (1024 threads):
//   1. radix select, four 8-bit digits from the top, finds the key T of the k-th smallest
//      entry and how many entries equal to T are still needed; keys live in shared memory
//      when the sequence fits (<= 16384 entries), otherwise every pass re-reads the scores;
//   2. one ordered pass collects every key < T and the first `need` keys == T (a block-wide
//      scan in index order gives each equal key its rank);
//   3. a bitonic sort of the <= 8192 selected (key << 32 | index) words puts them in order.
#include <algorithm>

#include "ptx.cuh"

namespace hss {
namespace {

constexpr int kThreads = 1024;
constexpr int kKeysCap = 16384;  // entries kept in shared memory

__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) u = 0x7F800000u;  // NaN ranks as +inf
    if (u == 0x80000000u) u = 0u;                          // -0 ranks as +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct RankShared {
    uint32_t hist[256];
    uint32_t warp_tot[32];
    uint32_t digit;
    uint32_t below;
    uint32_t count_sel;
    uint32_t eq_base;
};

__global__ void __launch_bounds__(kThreads, 1)
    rank_kernel(const float* __restrict__ scores, const int32_t* __restrict__ seq_offsets, int k,
                int sel_pow2, int32_t* __restrict__ victims) {
    extern __shared__ uint8_t smem_raw[];
    uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw);                      // [sel_pow2]
    RankShared* sh = reinterpret_cast<RankShared*>(sel + sel_pow2);
    uint32_t* keys = reinterpret_cast<uint32_t*>(sh + 1);                       // [kKeysCap]

    const int s = blockIdx.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t base = seq_offsets[s];
    const int n = static_cast<int>(seq_offsets[s + 1] - base);
    const int take = n < k ? n : k;
    int32_t* out = victims + static_cast<int64_t>(s) * k;
    const float* sc = scores + base;
    const bool in_smem = n <= kKeysCap;

    if (in_smem) {
        for (int i = tid; i < n; i += kThreads) keys[i] = score_key(sc[i]);
    }
    if (tid == 0) sh->count_sel = 0;
    __syncthreads();
    auto key_at = [&](int i) -> uint32_t { return in_smem ? keys[i] : score_key(__ldg(&sc[i])); };

    if (take < n) {
        // ---- 1. radix select of the take-th smallest key
        uint32_t prefix = 0, pmask = 0, need = static_cast<uint32_t>(take);
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            if (tid < 256) sh->hist[tid] = 0;
            __syncthreads();
            for (int i = tid; i < n; i += kThreads) {
                const uint32_t key = key_at(i);
                if ((key & pmask) == prefix) atomicAdd(&sh->hist[(key >> shift) & 0xFFu], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                uint32_t c[8], sum = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c[j] = sh->hist[lane * 8 + j];
                    sum += c[j];
                }
                uint32_t incl = sum;  // inclusive scan of the per-lane sums
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += v;
                }
                const uint32_t excl = incl - sum;
                // The digit bin is the first whose inclusive count reaches `need`.
                const bool mine = excl < need && need <= incl;
                if (mine) {
                    uint32_t run = excl;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (run + c[j] >= need) {
                            sh->digit = static_cast<uint32_t>(lane * 8 + j);
                            sh->below = run;
                            break;
                        }
                        run += c[j];
                    }
                }
            }
            __syncthreads();
            need -= sh->below;
            prefix |= sh->digit << shift;
            pmask |= 0xFFu << shift;
            __syncthreads();
        }
        const uint32_t T = prefix;

        // ---- 2. ordered collection: all keys < T, and the first `need` keys == T
        if (tid == 0) sh->eq_base = 0;
        __syncthreads();
        for (int c0 = 0; c0 < n; c0 += kThreads) {
            const int i = c0 + tid;
            const uint32_t key = i < n ? key_at(i) : 0xFFFFFFFFu;
            const bool lt = i < n && key < T;
            const bool eq = i < n && key == T;
            const uint32_t ball = __ballot_sync(0xffffffffu, eq);
            if (lane == 0) sh->warp_tot[warp] = __popc(ball);
            __syncthreads();
            uint32_t before = 0;
            for (int w = 0; w < warp; ++w) before += sh->warp_tot[w];
            const uint32_t rank_eq =
                sh->eq_base + before + __popc(ball & ((1u << lane) - 1u));
            if (lt || (eq && rank_eq < need)) {
                const uint32_t pos = atomicAdd(&sh->count_sel, 1u);
                if (pos < static_cast<uint32_t>(sel_pow2))
                    sel[pos] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(i);
            }
            __syncthreads();
            if (tid == 0) {
                uint32_t tot = 0;
                for (int w = 0; w < kThreads / 32; ++w) tot += sh->warp_tot[w];
                sh->eq_base += tot;
            }
            __syncthreads();
        }
    } else {
        for (int i = tid; i < n; i += kThreads)
            sel[i] = (static_cast<uint64_t>(key_at(i)) << 32) | static_cast<uint32_t>(i);
    }

    // ---- 3. bitonic sort of the selected words (padded to a power of two)
    int P = 1;
    while (P < take) P <<= 1;
    for (int i = take + tid; i < P; i += kThreads) sel[i] = ~0ull;
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < (P >> 1); t += kThreads) {
                const int i = 2 * t - (t & (stride - 1));
                const int j = i + stride;
                const uint64_t a = sel[i], b = sel[j];
                const bool asc = (i & size) == 0;
                if ((a > b) == asc) {
                    sel[i] = b;
                    sel[j] = a;
                }
            }
            __syncthreads();
        }
    }
    for (int j = tid; j < k; j += kThreads)
        out[j] = j < take ? static_cast<int32_t>(sel[j] & 0xFFFFFFFFull) : -1;
}

}  // namespace

hss_status launch_rank_victims(const float* scores, const int32_t* seq_offsets, int32_t num_seqs,
                               int64_t total, int32_t k, int32_t* victims, cudaStream_t stream) {
    (void)total;
    if (num_seqs == 0) return HSS_OK;
    const DeviceInfo* dev = current_device_info();
    if (dev == nullptr) return HSS_ERR_CUDA;
    int sel_pow2 = 1;
    while (sel_pow2 < k) sel_pow2 <<= 1;
    const int smem = sel_pow2 * 8 + static_cast<int>(sizeof(RankShared)) + kKeysCap * 4;
    static int set_bytes[64] = {0};
    const int d = dev->device & 63;
    if (set_bytes[d] < smem) {
        if (cudaFuncSetAttribute(rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return HSS_ERR_CUDA;
        set_bytes[d] = smem;
    }
    rank_kernel<<<num_seqs, kThreads, smem, stream>>>(scores, seq_offsets, k, sel_pow2, victims);
    return cudaGetLastError() == cudaSuccess ? HSS_OK : HSS_ERR_CUDA;
}

}  // namespace hss
