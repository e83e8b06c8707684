// rank_device.cuh -- per-sequence victim selection shared by the ranking kernel and the
// fused decode scorer.  See rank.cu for where it runs.
//
// Scores become order-preserving 32-bit keys (-0 -> +0, NaN -> +inf); the words
// (key << 32 | index) are unique, so "the k smallest, ascending, lower index first on ties"
// has exactly one answer.  One CTA ranks one sequence:
//   1. keys: held in registers (keys_per_thread per thread) when the sequence fits, otherwise
//      streamed from L2 in batches of eight independent loads per thread;
//   2. a block-wide min and max give the leading bits every key shares; radix select then
//      runs 8-bit digits from the first bit where keys differ, and stops as soon as the
//      chosen bin holds exactly the keys still needed (block scores cluster, so this skips
//      most of the passes a fixed 4 x 8-bit select would make);
//   3. collection: every key <= the threshold goes to the selection, placed by per-warp
//      ballot counts and one scan over the warps (streamed keys: warp-aggregated atomics);
//      the sort below orders ties by index.  When a mass of keys ties at the threshold and
//      they would not fit, an ordered pass takes the first ones by index instead;
//   4. a bitonic sort of the selected words: stages whose partner is in another warp go
//      through shared memory, stages within a warp run in registers with shuffles.
#pragma once

#include "ptx.cuh"

namespace hss {
namespace rankdev {

// Keys held in registers per thread: 16 at 256 threads, 8 at 1024 (64-register budget).
template <int THREADS>
__host__ __device__ constexpr int keys_per_thread() { return THREADS <= 256 ? 16 : 8; }

__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) u = 0x7F800000u;  // NaN ranks as +inf
    if (u == 0x80000000u) u = 0u;                          // -0 ranks as +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Keys of the order the selection works in: ascending scores (victims), or descending
// scores (DESC: the most relevant blocks first; NaN ranks like -inf, below every number).
// Either way the words (key << 32 | index) are then taken smallest first.
template <bool DESC>
__device__ __forceinline__ uint32_t rank_key(float f) {
    if constexpr (DESC) {
        if (f != f) f = -INFINITY;
        return ~score_key(f);
    } else {
        return score_key(f);
    }
}

struct RankShared {
    uint32_t hist[2][256];
    uint32_t red_min[32];
    uint32_t red_max[32];
    uint32_t warp_tot[32];
    uint32_t digit;
    uint32_t below;
    uint32_t bin_count;
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
    if (P <= THREADS) {
        // One element per thread.  Every thread runs the shuffle stages (threads past the end
        // hold the largest word), so no branch surrounds them.
        const bool act = tid < P;
        uint64_t v = act ? sel[tid] : ~0ull;
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1) v = cx_shfl(v, tid, stride, size);
        if (act) sel[tid] = v;
        __syncthreads();
        for (int size = 64; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride >= 32; stride >>= 1) {
                if (tid < (P >> 1)) {
                    const int i = 2 * tid - (tid & (stride - 1));
                    const int j = i + stride;
                    const uint64_t a = sel[i], b = sel[j];
                    if ((a > b) == ((i & size) == 0)) {
                        sel[i] = b;
                        sel[j] = a;
                    }
                }
                __syncthreads();
            }
            v = act ? sel[tid] : ~0ull;
#pragma unroll
            for (int stride = 16; stride > 0; stride >>= 1) v = cx_shfl(v, tid, stride, size);
            if (act) sel[tid] = v;
            __syncthreads();
        }
        return;
    }
    // Sizes up to 32: each warp's 32 consecutive elements sort in registers at once.
    for (int i = tid; i < P; i += THREADS) {
        uint64_t v = sel[i];
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
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
#pragma unroll
            for (int stride = 16; stride > 0; stride >>= 1) v = cx_shfl(v, i, stride, size);
            sel[i] = v;
        }
        __syncthreads();
    }
}

// The sequence's keys, seen in one of two ways.  Key i lives at (slot i / THREADS, thread
// i % THREADS), so a slot is a run of THREADS consecutive indices.
template <int THREADS, bool IN_REGS, bool DESC>
struct KeySet {
    const float* sc;
    int n;
    static constexpr int kKpt = keys_per_thread<THREADS>();
    uint32_t r[IN_REGS ? kKpt : 1];

    __device__ __forceinline__ void load(const float* s, int count) {
        sc = s;
        n = count;
        if constexpr (IN_REGS) {
#pragma unroll
            for (int j = 0; j < kKpt; ++j) {
                const int i = j * THREADS + static_cast<int>(threadIdx.x);
                r[j] = i < n ? rank_key<DESC>(__ldcg(&sc[i])) : 0u;
            }
        }
    }

    // fn(i, key) for every key this thread holds, in increasing index order.
    template <typename F>
    __device__ __forceinline__ void for_each(F&& fn) const {
        if constexpr (IN_REGS) {
#pragma unroll
            for (int j = 0; j < kKpt; ++j) {
                const int i = j * THREADS + static_cast<int>(threadIdx.x);
                if (i < n) fn(i, r[j]);
            }
        } else {
            for (int base = 0; base < n; base += 8 * THREADS) {
                uint32_t b[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {  // eight independent loads in flight
                    const int i = base + u * THREADS + static_cast<int>(threadIdx.x);
                    b[u] = i < n ? rank_key<DESC>(__ldcg(&sc[i])) : 0u;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = base + u * THREADS + static_cast<int>(threadIdx.x);
                    if (i < n) fn(i, b[u]);
                }
            }
        }
    }

    // The key of index i held by this thread in slot j (i = j * THREADS + tid), or the
    // sentinel when i >= n.  Used by the ordered pass, which walks slots in index order.
    __device__ __forceinline__ uint32_t slot_key(int j) const {
        const int i = j * THREADS + static_cast<int>(threadIdx.x);
        if (i >= n) return 0xFFFFFFFFu;
        if constexpr (IN_REGS) {
            uint32_t v = 0;
#pragma unroll
            for (int q = 0; q < kKpt; ++q)
                if (q == j) v = r[q];
            return v;
        } else {
            return rank_key<DESC>(__ldcg(&sc[i]));
        }
    }
};

template <int THREADS, bool IN_REGS, bool DESC>
__device__ void rank_with(const float* __restrict__ sc, int n, int k, int32_t* __restrict__ out,
                          uint64_t* sel, int sel_cap, RankShared* sh) {
    constexpr int kWarps = THREADS / 32;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t lane_lt = (1u << lane) - 1u;
    const int take = n < k ? n : k;

    KeySet<THREADS, IN_REGS, DESC> ks;
    ks.load(sc, n);  // the loads are in flight while the histograms are cleared
    if (tid < 256) {
        sh->hist[0][tid] = 0;
        sh->hist[1][tid] = 0;
    }
    if (tid == 0) sh->count_sel = 0;
    __syncthreads();  // the zeroed histogram and counter before anyone adds to them

    // Warp-aggregated append of (key, index) to sel.
    auto append = [&](bool pick, uint32_t key, int i) {
        const uint32_t ball = __ballot_sync(0xffffffffu, pick);
        uint32_t wbase = 0;
        if (lane == 0 && ball) wbase = atomicAdd(&sh->count_sel, __popc(ball));
        wbase = __shfl_sync(0xffffffffu, wbase, 0);
        if (pick) {
            const uint32_t pos = wbase + __popc(ball & lane_lt);
            if (pos < static_cast<uint32_t>(sel_cap))
                sel[pos] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(i);
        }
    };
    // Every lane of every warp walks the same number of rounds, so the ballots are full.
    auto for_each_uniform = [&](auto&& fn) {
        const int rounds = (n + THREADS - 1) / THREADS;
        if constexpr (IN_REGS) {
#pragma unroll
            for (int j = 0; j < KeySet<THREADS, IN_REGS, DESC>::kKpt; ++j) {
                if (j < rounds) {
                    const int i = j * THREADS + tid;
                    fn(i < n, i < n ? ks.r[j] : 0u, i);
                }
            }
        } else {
            for (int j = 0; j < rounds; ++j) {
                const int i = j * THREADS + tid;
                fn(i < n, ks.slot_key(j), i);
            }
        }
    };

    // Every key with pred(key) goes to sel.  With the keys in registers the positions come
    // from per-warp ballot counts and one scan over the warps (no atomics, one barrier);
    // streamed keys use the warp-aggregated append.  The order in sel is irrelevant: the
    // words are sorted afterwards.
    auto collect = [&](auto&& pred) {
        if constexpr (IN_REGS) {
            constexpr int kK = KeySet<THREADS, IN_REGS, DESC>::kKpt;
            // The ballots are taken twice (count, then place) rather than kept in registers.
            // No branch around them: `i < n` already drops the slots past the end, and a
            // ballot under a condition costs a reconvergence point per slot.
            uint32_t wcount = 0;
#pragma unroll
            for (int j = 0; j < kK; ++j) {
                const int i = j * THREADS + tid;
                wcount += __popc(__ballot_sync(0xffffffffu, i < n && pred(ks.r[j])));
            }
            if (lane == 0) sh->warp_tot[warp] = wcount;
            __syncthreads();
            uint32_t base = 0;
            for (int w = 0; w < warp; ++w) base += sh->warp_tot[w];
#pragma unroll
            for (int j = 0; j < kK; ++j) {
                const int i = j * THREADS + tid;
                const bool pick = i < n && pred(ks.r[j]);
                const uint32_t ball = __ballot_sync(0xffffffffu, pick);
                const uint32_t pos = base + __popc(ball & lane_lt);
                if (pick && pos < static_cast<uint32_t>(sel_cap))
                    sel[pos] = (static_cast<uint64_t>(ks.r[j]) << 32) | static_cast<uint32_t>(i);
                base += __popc(ball);
            }
        } else {
            for_each_uniform([&](bool valid, uint32_t key, int i) {
                append(valid && pred(key), key, i);
            });
        }
    };

    int count = 0;  // words placed in sel
    if (take < n) {
        // ---- 1. the bits every key shares
        uint32_t mn = 0xFFFFFFFFu, mx = 0u;
        ks.for_each([&](int, uint32_t key) {
            mn = key < mn ? key : mn;
            mx = key > mx ? key : mx;
        });
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const uint32_t a = __shfl_xor_sync(0xffffffffu, mn, off);
            const uint32_t b = __shfl_xor_sync(0xffffffffu, mx, off);
            mn = a < mn ? a : mn;
            mx = b > mx ? b : mx;
        }
        if (lane == 0) {
            sh->red_min[warp] = mn;
            sh->red_max[warp] = mx;
        }
        __syncthreads();
        mn = 0xFFFFFFFFu;
        mx = 0u;
        for (int w = 0; w < kWarps; ++w) {
            mn = sh->red_min[w] < mn ? sh->red_min[w] : mn;
            mx = sh->red_max[w] > mx ? sh->red_max[w] : mx;
        }

        uint32_t T;          // threshold: the selection is every key <= T (+ tie handling)
        int n_lt, n_eq;      // keys below T, keys equal to T (n_eq = 0: no ties to resolve)
        uint32_t need = static_cast<uint32_t>(take);
        if (mn == mx) {
            T = mn;
            n_lt = 0;
            n_eq = n;
        } else {
            // ---- 2. radix select from the highest differing bit, 8 bits at a time
            int hi = 31 - __clz(mn ^ mx);
            const uint32_t free_bits = hi == 31 ? 0xFFFFFFFFu : ((2u << hi) - 1u);
            uint32_t pmask = ~free_bits;
            uint32_t prefix = mn & pmask;
            bool exact = false;
            int pass = 0;
            while (hi >= 0) {
                const int lo = hi >= 7 ? hi - 7 : 0;
                const uint32_t wmask = (2u << (hi - lo)) - 1u;
                uint32_t* H = sh->hist[pass & 1];
                ks.for_each([&](int, uint32_t key) {
                    if ((key & pmask) == prefix) atomicAdd(&H[(key >> lo) & wmask], 1u);
                });
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
                    if (excl < need && need <= incl) {  // the bin where the count reaches need
                        uint32_t run = excl;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (run + c[j] >= need) {
                                sh->digit = static_cast<uint32_t>(lane * 8 + j);
                                sh->below = run;
                                sh->bin_count = c[j];
                                break;
                            }
                            run += c[j];
                        }
                    }
                }
                __syncthreads();
                need -= sh->below;
                prefix |= sh->digit << lo;
                pmask |= wmask << lo;
                ++pass;
                if (sh->bin_count == need) {  // the whole bin is taken: no finer digit needed
                    exact = true;
                    T = prefix | (lo > 0 ? (1u << lo) - 1u : 0u);
                    break;
                }
                hi = lo - 1;
            }
            if (exact) {
                n_lt = take;
                n_eq = 0;
            } else {
                T = prefix;
                n_lt = take - static_cast<int>(need);
                n_eq = static_cast<int>(sh->bin_count);
            }
        }

        if (n_lt + n_eq <= sel_cap) {
            // ---- 3a. every key <= T; the sort orders ties at T by index
            collect([&](uint32_t key) { return key <= T; });
            count = n_lt + n_eq;
        } else {
            // ---- 3b. ordered: keys < T, then the first `need` keys == T by index
            if (tid == 0) sh->eq_base = 0;
            __syncthreads();
            for_each_uniform([&](bool valid, uint32_t key, int i) {
                const bool lt = valid && key < T;
                const bool eq = valid && key == T;
                const uint32_t ball_eq = __ballot_sync(0xffffffffu, eq);
                if (lane == 0) sh->warp_tot[warp] = __popc(ball_eq);
                __syncthreads();
                uint32_t before = 0;
                for (int w = 0; w < warp; ++w) before += sh->warp_tot[w];
                const uint32_t rank_eq = sh->eq_base + before + __popc(ball_eq & lane_lt);
                append(lt || (eq && rank_eq < need), key, i);
                __syncthreads();
                if (tid == 0) {
                    uint32_t tot = 0;
                    for (int w = 0; w < kWarps; ++w) tot += sh->warp_tot[w];
                    sh->eq_base += tot;
                }
                __syncthreads();
            });
            count = take;
        }
    } else {
        collect([](uint32_t) { return true; });
        count = n;
    }

    // ---- 4. sort the selected words (padded to a power of two).  count never exceeds the
    // buffer when the histograms are consistent; the clamp keeps every access inside it
    // regardless.
    if (count > sel_cap) count = sel_cap;
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

// Ranks one sequence: victims out[0, k) of the n scores sc[0, n).  Every thread of the CTA
// calls it (THREADS = blockDim.x); sel [sel_cap] and sh are shared memory.  Scores are read
// through L2 (ld.global.cg), so the function may also run in the kernel that wrote them,
// after a fence.
template <int THREADS, bool DESC = false>
__device__ void rank_sequence(const float* __restrict__ sc, int n, int k,
                              int32_t* __restrict__ out, uint64_t* sel, int sel_cap,
                              RankShared* sh) {
    if (n <= THREADS * keys_per_thread<THREADS>())
        rank_with<THREADS, true, DESC>(sc, n, k, out, sel, sel_cap, sh);
    else
        rank_with<THREADS, false, DESC>(sc, n, k, out, sel, sel_cap, sh);
}

// Shared-memory bytes rank_sequence needs.
inline int rank_smem_bytes(int sel_cap) {
    return sel_cap * 8 + static_cast<int>(sizeof(RankShared));
}

inline int rank_sel_cap(int k) {
    int pow2k = 1;
    while (pow2k < k) pow2k <<= 1;
    return 2 * pow2k;  // room for every key <= T when there are some ties at the cutoff
}

}  // namespace rankdev
}  // namespace hss
