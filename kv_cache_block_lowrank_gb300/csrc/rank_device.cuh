// rank_device.cuh -- per-sequence victim selection shared by the ranking kernel and the
// fused decode scorer: radix select of the k smallest order-preserving keys, collection,
// and a bitonic sort of the (key << 32 | index) words.  See rank.cu for the design.
#pragma once

#include "ptx.cuh"

namespace hss {
namespace rankdev {

constexpr int kKeysCap = 16384;

__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) u = 0x7F800000u;  // NaN ranks as +inf
    if (u == 0x80000000u) u = 0u;                          // -0 ranks as +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct RankShared {
    uint32_t hist[2][256];
    uint32_t warp_tot[32];
    uint32_t digit;
    uint32_t below;
    uint32_t eq_count;
    uint32_t count_sel;
    uint32_t eq_base;
};

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v), m);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), m);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Compare-exchange of element i with element i ^ stride inside one warp (all lanes take part).
__device__ __forceinline__ uint64_t cx_shfl(uint64_t v, int i, int stride, int size) {
    const uint64_t o = shfl_xor_u64(v, stride);
    const bool asc = (i & size) == 0;
    const bool lower = (i & stride) == 0;
    return (lower == asc) ? (v < o ? v : o) : (v < o ? o : v);
}

// Ascending bitonic sort of sel[0, P), P a power of two.  All THREADS threads call it.
template <int THREADS>
__device__ void bitonic_sort(uint64_t* sel, int P) {
    const int tid = threadIdx.x;
    if (P <= 1) return;
    if (P < 32) {
        if (tid < 32) {
            uint64_t v = tid < P ? sel[tid] : ~0ull;
            for (int size = 2; size <= 32; size <<= 1)
                for (int stride = size >> 1; stride > 0; stride >>= 1)
                    v = cx_shfl(v, tid, stride, size);
            if (tid < P) sel[tid] = v;
        }
        __syncthreads();
        return;
    }
    // Sizes up to 32: each warp's 32 consecutive elements sort in registers at once.
    for (int i = tid; i < P; i += THREADS) {
        uint64_t v = sel[i];
        for (int size = 2; size <= 32; size <<= 1)
            for (int stride = size >> 1; stride > 0; stride >>= 1) v = cx_shfl(v, i, stride, size);
        sel[i] = v;
    }
    __syncthreads();
    for (int size = 64; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride >= 32; stride >>= 1) {
            for (int t = tid; t < (P >> 1); t += THREADS) {
                const int i = 2 * t - (t & (stride - 1));
                const int j = i + stride;
                const uint64_t a = sel[i], b = sel[j];
                if ((a > b) == ((i & size) == 0)) {
                    sel[i] = b;
                    sel[j] = a;
                }
            }
            __syncthreads();
        }
        for (int i = tid; i < P; i += THREADS) {
            uint64_t v = sel[i];
            for (int stride = 16; stride > 0; stride >>= 1) v = cx_shfl(v, i, stride, size);
            sel[i] = v;
        }
        __syncthreads();
    }
}

// Ranks one sequence: victims out[0, k) of the n scores sc[0, n).  Every thread of the CTA
// calls it (THREADS = blockDim.x); sel [sel_cap], sh and keys [keys_cap] are shared memory.
// Scores are read through L2 (ld.global.cg), so the function may also run in the kernel
// that wrote them, after a fence.
template <int THREADS>
__device__ void rank_sequence(const float* __restrict__ sc, int n, int k,
                              int32_t* __restrict__ out, uint64_t* sel, int sel_cap,
                              RankShared* sh, uint32_t* keys, int keys_cap) {
    constexpr int kWarps = THREADS / 32;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t lane_lt = (1u << lane) - 1u;

    if (tid < 256) {
        sh->hist[0][tid] = 0;
        sh->hist[1][tid] = 0;
    }
    if (tid == 0) sh->count_sel = 0;
    const int take = n < k ? n : k;
    const bool in_smem = n <= keys_cap;

    if (in_smem) {
        for (int i = tid; i < n; i += THREADS) keys[i] = score_key(__ldcg(&sc[i]));
    }
    __syncthreads();
    auto key_at = [&](int i) -> uint32_t { return in_smem ? keys[i] : score_key(__ldcg(&sc[i])); };
    int count = 0;  // words placed in sel
    if (take < n) {
        // ---- 1. radix select
        uint32_t prefix = 0, pmask = 0, need = static_cast<uint32_t>(take);
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            uint32_t* H = sh->hist[pass & 1];
            for (int i = tid; i < n; i += THREADS) {
                const uint32_t key = key_at(i);
                if ((key & pmask) == prefix) atomicAdd(&H[(key >> shift) & 0xFFu], 1u);
            }
            if (tid < 256) sh->hist[(pass & 1) ^ 1][tid] = 0;
            __syncthreads();
            if (warp == 0) {
                uint32_t c[8], sum = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c[j] = H[lane * 8 + j];
                    sum += c[j];
                }
                uint32_t incl = sum;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += v;
                }
                const uint32_t excl = incl - sum;
                if (excl < need && need <= incl) {  // the bin where the count reaches `need`
                    uint32_t run = excl;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (run + c[j] >= need) {
                            sh->digit = static_cast<uint32_t>(lane * 8 + j);
                            sh->below = run;
                            sh->eq_count = c[j];
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
        }
        const uint32_t T = prefix;
        const int n_lt = take - static_cast<int>(need);
        const int n_eq = static_cast<int>(sh->eq_count);

        if (n_lt + n_eq <= sel_cap) {
            // ---- 2a. every key <= T; the sort orders ties at T by index
            for (int c0 = 0; c0 < n; c0 += THREADS) {
                const int i = c0 + tid;
                const uint32_t key = i < n ? key_at(i) : 0xFFFFFFFFu;
                const bool pick = i < n && key <= T;
                const uint32_t ball = __ballot_sync(0xffffffffu, pick);
                uint32_t wbase = 0;
                if (lane == 0 && ball) wbase = atomicAdd(&sh->count_sel, __popc(ball));
                wbase = __shfl_sync(0xffffffffu, wbase, 0);
                if (pick) {
                    const uint32_t pos = wbase + __popc(ball & lane_lt);
                    if (pos < static_cast<uint32_t>(sel_cap))
                        sel[pos] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(i);
                }
            }
            count = n_lt + n_eq;
        } else {
            // ---- 2b. ordered: keys < T, then the first `need` keys == T by index
            if (tid == 0) sh->eq_base = 0;
            __syncthreads();
            for (int c0 = 0; c0 < n; c0 += THREADS) {
                const int i = c0 + tid;
                const uint32_t key = i < n ? key_at(i) : 0xFFFFFFFFu;
                const bool lt = i < n && key < T;
                const bool eq = i < n && key == T;
                const uint32_t ball_eq = __ballot_sync(0xffffffffu, eq);
                if (lane == 0) sh->warp_tot[warp] = __popc(ball_eq);
                __syncthreads();
                uint32_t before = 0;
                for (int w = 0; w < warp; ++w) before += sh->warp_tot[w];
                const uint32_t rank_eq = sh->eq_base + before + __popc(ball_eq & lane_lt);
                const bool pick = lt || (eq && rank_eq < need);
                const uint32_t ball = __ballot_sync(0xffffffffu, pick);
                uint32_t wbase = 0;
                if (lane == 0 && ball) wbase = atomicAdd(&sh->count_sel, __popc(ball));
                wbase = __shfl_sync(0xffffffffu, wbase, 0);
                if (pick) {
                    const uint32_t pos = wbase + __popc(ball & lane_lt);
                    if (pos < static_cast<uint32_t>(sel_cap))
                        sel[pos] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(i);
                }
                __syncthreads();
                if (tid == 0) {
                    uint32_t tot = 0;
                    for (int w = 0; w < kWarps; ++w) tot += sh->warp_tot[w];
                    sh->eq_base += tot;
                }
                __syncthreads();
            }
            count = take;
        }
    } else {
        for (int i = tid; i < n; i += THREADS)
            sel[i] = (static_cast<uint64_t>(key_at(i)) << 32) | static_cast<uint32_t>(i);
        count = n;
    }

    // ---- 3. sort the selected words (padded to a power of two)
    int P = 1;
    while (P < count) P <<= 1;
    __syncthreads();
    for (int i = count + tid; i < P; i += THREADS) sel[i] = ~0ull;
    __syncthreads();
    bitonic_sort<THREADS>(sel, P);
    for (int j = tid; j < k; j += THREADS)
        out[j] = j < take ? static_cast<int32_t>(sel[j] & 0xFFFFFFFFull) : -1;
    __syncthreads();
}

// Shared-memory bytes rank_sequence needs for a given k and key cache size.
inline int rank_smem_bytes(int sel_cap, int keys_cap) {
    return sel_cap * 8 + static_cast<int>(sizeof(RankShared)) + keys_cap * 4;
}

inline int rank_sel_cap(int k) {
    int pow2k = 1;
    while (pow2k < k) pow2k <<= 1;
    return 2 * pow2k;  // room for every key <= T when there are some ties at the cutoff
}

}  // namespace rankdev
}  // namespace hss
