// score_tc.cu -- block scores for prefill chunks on the 5th-generation tensor cores.
//
// Page "metrale_storage/predictor.rs", Predictor::score_blocks: a block's score is the max,
// over query heads and tokens, of the projected dot product Qp . A_g (query head h reads kv
// head h / g).  With a prefill chunk of R query rows there are R * g query vectors per kv
// head, and Qp . A_g^T becomes a real dense contraction (R * g x tokens x r per kv head), so
// it runs on tcgen05.mma with TMEM accumulators.
//
// Orientation: tokens are the M side (128-token tiles = 128 / block_size blocks of one kv
// head, gathered through the block table with one TMA box per block), query vectors the N
// side, r the K side.  Then every TMEM lane (= thread in the epilogue) holds one token's
// dot products with 256 query vectors: the max over query vectors is a per-thread register
// reduction, and the max over a block's tokens is a 16-lane shuffle reduction.
//
// Work units: (sequence s, kv head c, 128-token tile) for one slice of up to 1024 query
// vectors.  CTAs come in groups of `nslices`, one CTA per slice; the CTAs of a group walk the
// same contiguous run of (s, c, tile) units in step, so each A tile is fetched from HBM once
// and served from L2 to the group's other slices.  A CTA's slice of Qp stays resident in
// shared memory (B operand, K-major, swizzled) and is reloaded only when its run crosses into
// the next (s, c).  Roles (persistent, 1 CTA per SM):
//   warp 0      TMA producer (Qp slices; per-block A_g boxes into a ring of stages)
//   warp 1      TMEM allocator (512 columns) and MMA issuer, M=128, N=256, K=16 steps
//   warps 2..9  epilogue, two warpgroups that each drain half (128 columns) of every
//               256-column accumulator chunk: four 32-column tcgen05.ld per wait, 3-input
//               max, block max by shuffles, one float atomic max per block and warpgroup
// Scores are first set to -inf (separate tiny kernel); every unit atomically maxes its
// partial block maximum into the block's score.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "ptx.cuh"

namespace hss {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

constexpr int kThreads = 320;  // producer warp, MMA warp, two epilogue warpgroups
constexpr int kTileTokens = 128;     // UMMA M
constexpr int kNChunk = 256;         // UMMA N per accumulator buffer
constexpr int kMaxSliceVecs = 1024;  // query vectors resident per slice
constexpr int kMaxSeqs = 1024;       // prefix table of units per sequence lives in smem
constexpr int kBudgetB = 128 * 1024;

struct TcLayout {
    int row_bytes;      // bytes of one swizzled row segment: min(r, 64) * 2
    int kchunks;        // r / (row_bytes / 2)
    int slice;          // query vectors per slice (multiple of 256)
    int b_bytes;        // slice * r * 2
    int a_stage_bytes;  // 128 * r * 2
    int stages;
    int total_bytes;
};

TcLayout make_tc_layout(int r, int smem_budget) {
    TcLayout L;
    L.row_bytes = (r >= 64 ? 64 : r) * 2;
    L.kchunks = r * 2 / L.row_bytes;
    int slice = kBudgetB / (r * 2);
    slice = slice / kNChunk * kNChunk;
    L.slice = std::min(kMaxSliceVecs, std::max(kNChunk, slice));
    L.b_bytes = L.slice * r * 2;
    L.a_stage_bytes = kTileTokens * r * 2;
    // barriers (512) + units before each sequence (int64) + sequence offsets (int32)
    const int fixed = 1024 + 512 + (kMaxSeqs + 1) * 8 + (kMaxSeqs + 1) * 4 + L.b_bytes;
    L.stages = std::min(4, (smem_budget - fixed) / L.a_stage_bytes);
    L.total_bytes = fixed + L.stages * L.a_stage_bytes;
    return L;
}

struct TcParams {
    const int32_t* table;
    const int32_t* seq_offsets;
    float* scores;
    int32_t* dev_status;
    int32_t* lib_error;
    int64_t layer_slots;  // layer * max_blocks
    int64_t max_blocks;
    int64_t units_per_group;  // (s, c, tile) units per CTA group
    int32_t num_groups;       // CTA groups; CTA b works on slice b % nslices of group b / nslices
    int32_t num_seqs;
    int32_t nkv;
    int32_t g;
    int32_t bs;
    int32_t r;
    int32_t rows;  // query rows per sequence
    int32_t nvec;  // rows * g query vectors per (sequence, kv head)
    int32_t nslices;
    int32_t slice;
    int32_t bpt;  // blocks per 128-token tile
    int32_t row_bytes;
    int32_t kchunks;
    int32_t b_bytes;
    int32_t a_stage_bytes;
    int32_t stages;
};

struct Unit {
    int s, c, q;
    int64_t t;       // tile within the sequence
    int64_t tiles;   // the sequence's tiles
    int64_t first;   // table index of the sequence's first block
    int64_t end;     // one past its last
    int64_t pair;    // (s, c, q) identity
};

// Unit u -> (sequence, kv head, tile) for slice q, with units_before[s] = units of
// sequences before s and offs = the sequence offsets, both cached in shared memory.
__device__ __forceinline__ Unit decode_unit(int64_t u, int q, const TcParams& p,
                                            const int64_t* units_before, const int32_t* offs) {
    int lo = 0, hi = p.num_seqs;  // last s with units_before[s] <= u
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (units_before[mid] <= u) lo = mid; else hi = mid;
    }
    Unit x;
    x.s = lo;
    x.first = offs[lo];
    x.end = offs[lo + 1];
    const int64_t tiles = (x.end - x.first + p.bpt - 1) / p.bpt;
    x.tiles = tiles;
    const int64_t local = u - units_before[lo];
    const int64_t c = local / tiles;
    x.t = local - c * tiles;
    x.c = static_cast<int>(c);
    x.q = q;
    x.pair = units_before[lo] + c * tiles;  // unique per (s, c); the slice is fixed per CTA
    return x;
}

// The unit after x (u + 1): the next tile, kv head or non-empty sequence, without
// decode_unit's search and 64-bit divisions (the single MMA-issuing thread pays them per
// tile otherwise).  Past the last unit it leaves x on the last sequence; nobody reads it.
__device__ __forceinline__ void advance_unit(Unit& x, const TcParams& p,
                                             const int64_t* units_before, const int32_t* offs) {
    if (++x.t < x.tiles) return;
    x.t = 0;
    if (++x.c < p.nkv) {
        x.pair += x.tiles;
        return;
    }
    x.c = 0;
    int s = x.s + 1;
    if (s >= p.num_seqs) return;
    while (s + 1 < p.num_seqs && units_before[s + 1] == units_before[s]) ++s;  // empty ones
    x.s = s;
    x.first = offs[s];
    x.end = offs[s + 1];
    x.tiles = (x.end - x.first + p.bpt - 1) / p.bpt;
    x.pair = units_before[s];
}

__device__ __forceinline__ void atomic_max_f32(float* addr, float v) {
    v = v + 0.0f;  // -0 -> +0, so the integer orderings below agree with the float order
    if (v >= 0.0f) {
        atomicMax(reinterpret_cast<int*>(addr), __float_as_int(v));
    } else {
        atomicMin(reinterpret_cast<unsigned int*>(addr), __float_as_uint(v));
    }
}

__global__ void fill_neg_inf(float* __restrict__ x, int64_t n) {
    grid_dependency_wait();
    grid_launch_dependents();
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        x[i] = -INFINITY;
}

// Per-row scores (ROWG = g > 0): a thread takes one token's dot products with 32 query
// vectors (32 / g query rows) at a time.  After the max over each row's g heads, a reduce-scatter over
// the block's lanes leaves every lane with whole-block maxima of distinct rows:
// at each step the lanes whose mask bit is set keep the upper half of their list and take
// the partner's upper half, the others the lower half; once one value is left the remaining
// steps are plain max reductions.
template <int N, int CNT, int M>
__device__ __forceinline__ void reduce_scatter(float (&x)[N], int lane) {
    if constexpr (M > 0) {
        if constexpr (CNT > 1) {
            constexpr int H = CNT / 2;
            const bool upper = (lane & M) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = upper ? x[i] : x[i + H];
                const float keep = upper ? x[i + H] : x[i];
                x[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, M));
            }
            reduce_scatter<N, H, M / 2>(x, lane);
        } else {
            x[0] = fmaxf(x[0], __shfl_xor_sync(0xffffffffu, x[0], M));
            reduce_scatter<N, 1, M / 2>(x, lane);
        }
    }
}

// Row maxima of the COLS columns v[OFF .. OFF + COLS - 1] (vectors v0 .. v0 + COLS - 1, the
// first `valid` real)
// for the tokens of one block (BS lanes), max-combined into scores[row * stride + e].
template <int G, int BS, int OFF, int COLS>
__device__ __forceinline__ void rows_to_scores(const uint32_t (&v)[128], int valid, int v0,
                                               int lane, int rows, float* __restrict__ scores,
                                               int64_t stride, int64_t e, bool e_ok) {
    constexpr int V = COLS / G;
    float x[V];
    if (valid >= COLS) {  // every column real: a plain 3-input max tree per row
#pragma unroll
        for (int i = 0; i < V; ++i) {
            float m = __uint_as_float(v[OFF + i * G]);
#pragma unroll
            for (int j = 1; j < G; j += 2)
                m = j + 1 < G ? fmax3(m, __uint_as_float(v[OFF + i * G + j]),
                                      __uint_as_float(v[OFF + i * G + j + 1]))
                              : fmaxf(m, __uint_as_float(v[OFF + i * G + j]));
            x[i] = m;
        }
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) {
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < G; ++j)
                if (i * G + j < valid) m = fmaxf(m, __uint_as_float(v[OFF + i * G + j]));
            x[i] = m;
        }
    }
    reduce_scatter<V, V, BS / 2>(x, lane);
    constexpr int LOGV = V >= 32 ? 5 : V >= 16 ? 4 : V >= 8 ? 3 : V >= 4 ? 2 : V >= 2 ? 1 : 0;
    static_assert(V <= 32, "at most 32 row values per lane");
    constexpr int LOGB = BS == 32 ? 5 : 4;
    constexpr int S = LOGV < LOGB ? LOGV : LOGB;  // scatter steps
    constexpr int LEFT = V >> S;                  // values per lane at the end
    const int lb = lane & (BS - 1);
    if (!e_ok || (lb & ((1 << (LOGB - S)) - 1)) != 0) return;  // one writer per value
    const int sel = lb >> (LOGB - S);
#pragma unroll
    for (int i = 0; i < LEFT; ++i) {
        const int row = v0 / G + sel * LEFT + i;
        if (row < rows) atomic_max_f32(scores + row * stride + e, x[i]);
    }
}

// Max over each row's G heads for 64 columns va[0 .. 63] (the first `valid` real) into
// x[XOFF .. XOFF + 64 / G).
template <int G, int XOFF, int V>
__device__ __forceinline__ void group_max64(const uint32_t (&va)[64], int valid, float (&x)[V]) {
    constexpr int R = 64 / G;
    if (valid >= 64) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float m = __uint_as_float(va[i * G]);
#pragma unroll
            for (int j = 1; j < G; j += 2)
                m = j + 1 < G ? fmax3(m, __uint_as_float(va[i * G + j]),
                                      __uint_as_float(va[i * G + j + 1]))
                              : fmaxf(m, __uint_as_float(va[i * G + j]));
            x[XOFF + i] = m;
        }
    } else {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < G; ++j)
                if (i * G + j < valid) m = fmaxf(m, __uint_as_float(va[i * G + j]));
            x[XOFF + i] = m;
        }
    }
}

// Whole-block maxima of the V row values x (rows v0 / G ..): reduce-scatter over the block's
// BS lanes, then one float atomic max per value into scores[row * stride + e].
template <int G, int BS, int V>
__device__ __forceinline__ void scatter_rows(float (&x)[V], int v0, int lane, int rows,
                                             float* __restrict__ scores, int64_t stride,
                                             int64_t e, bool e_ok) {
    reduce_scatter<V, V, BS / 2>(x, lane);
    constexpr int LOGV = V >= 32 ? 5 : V >= 16 ? 4 : V >= 8 ? 3 : V >= 4 ? 2 : V >= 2 ? 1 : 0;
    static_assert(V <= 32, "at most 32 row values per lane");
    constexpr int LOGB = BS == 32 ? 5 : 4;
    constexpr int S = LOGV < LOGB ? LOGV : LOGB;
    constexpr int LEFT = V >> S;
    const int lb = lane & (BS - 1);
    if (!e_ok || (lb & ((1 << (LOGB - S)) - 1)) != 0) return;
    const int sel = lb >> (LOGB - S);
#pragma unroll
    for (int i = 0; i < LEFT; ++i) {
        const int row = v0 / G + sel * LEFT + i;
        if (row < rows) atomic_max_f32(scores + row * stride + e, x[i]);
    }
}

// MASKED: the call passed ctx_len or row_pos0.  A template parameter, so the unmasked kernel
// carries none of the mask arithmetic.  The mask pointers are kernel arguments of their own:
// two more fields in TcParams made the unmasked kernel 7% slower on GB300.
// ROWG > 0: per-row scores (one sequence; g = ROWG query heads per kv head): scores is
// [rows, total] and receives the max over heads and tokens for every (row, block).
template <bool MASKED, int ROWG>
__global__ void __launch_bounds__(kThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_q, const TcParams p,
                    const int32_t* __restrict__ ctx_len, const int32_t* __restrict__ row_pos0,
                    const int64_t one_total) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sB = smem;
    uint8_t* sA = sB + p.b_bytes;
    uint64_t* a_full = reinterpret_cast<uint64_t*>(sA + p.stages * p.a_stage_bytes);
    uint64_t* a_empty = a_full + p.stages;
    uint64_t* b_full = a_empty + p.stages;
    uint64_t* b_empty = b_full + 1;
    uint64_t* t_full = b_empty + 1;
    uint64_t* t_empty = t_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + 2);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    int64_t* units_before = reinterpret_cast<int64_t*>(smem + p.b_bytes +
                                                       p.stages * p.a_stage_bytes + 512);
    int32_t* offs = reinterpret_cast<int32_t*>(units_before + p.num_seqs + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr uint32_t kTmemCols = 512;

    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    grid_dependency_wait();
    grid_launch_dependents();
    // Units before each sequence: nkv * nslices * tiles(s) per sequence.
    if (threadIdx.x == 0) {
        int64_t acc = 0;
        for (int s = 0; s < p.num_seqs; ++s) {
            units_before[s] = acc;
            // No offsets array: one sequence of `one_total` entries.
            offs[s] = p.seq_offsets != nullptr ? p.seq_offsets[s] : 0;
            const int64_t n = p.seq_offsets != nullptr
                                  ? static_cast<int64_t>(p.seq_offsets[s + 1]) - p.seq_offsets[s]
                                  : one_total;
            acc += static_cast<int64_t>(p.nkv) * ((n + p.bpt - 1) / p.bpt);
        }
        units_before[p.num_seqs] = acc;
        offs[p.num_seqs] = p.seq_offsets != nullptr ? p.seq_offsets[p.num_seqs] : one_total;
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        mbar_init(b_full, 1);
        mbar_init(b_empty, 1);
        for (int a = 0; a < 2; ++a) {
            mbar_init(&t_full[a], 1);
            mbar_init(&t_empty[a], 8);  // every epilogue warp drains part of each chunk
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    // CTA b serves slice q = b % nslices for the units of group b / nslices.  The host sized
    // the groups from an upper bound; the exact unit count is units_before[num_seqs].
    const int q_slice = static_cast<int>(blockIdx.x % p.nslices);
    const int64_t group = blockIdx.x / p.nslices;
    const int64_t u_begin = group < p.num_groups ? group * p.units_per_group : 0;
    const int64_t u_end = group < p.num_groups
                              ? min(units_before[p.num_seqs], u_begin + p.units_per_group)
                              : 0;
    const int nchunks = p.slice / kNChunk;
    const int elems_per_row = p.row_bytes / 2;
    Unit first_unit{};
    if (u_begin < u_end) first_unit = decode_unit(u_begin, q_slice, p, units_before, offs);

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmap_a);
            tma_prefetch_desc(&tmap_q);
            int stage = 0;
            uint32_t phase = 0, b_empty_phase = 0, b_loads = 0;
            int64_t prev_pair = -1, issued = 0;
            bool ok = true;
            Unit x = first_unit;
            for (int64_t u = u_begin; u < u_end && ok;
                 ++u, advance_unit(x, p, units_before, offs)) {
                if (x.pair != prev_pair) {
                    if (prev_pair >= 0) {
                        ok = mbar_wait(b_empty, b_empty_phase);
                        b_empty_phase ^= 1u;
                        if (!ok) break;
                    }
                    mbar_arrive_expect_tx(b_full, static_cast<uint32_t>(p.b_bytes));
                    for (int kc = 0; kc < p.kchunks; ++kc) {
                        for (int j = 0; j < nchunks; ++j) {
                            const int64_t z = static_cast<int64_t>(x.s) * p.rows +
                                              (static_cast<int64_t>(x.q) * p.slice +
                                               j * kNChunk) / p.g;
                            tma_load_3d(sB + kc * (p.slice * p.row_bytes) +
                                            j * (kNChunk * p.row_bytes),
                                        &tmap_q, b_full, kc * elems_per_row, x.c * p.g,
                                        static_cast<int32_t>(z));
                        }
                    }
                    ++b_loads;
                    prev_pair = x.pair;
                }
                if (!mbar_wait(&a_empty[stage], phase ^ 1u) || *(volatile int*)abort_flag) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&a_full[stage], static_cast<uint32_t>(p.a_stage_bytes));
                uint8_t* dst = sA + stage * p.a_stage_bytes;
                for (int blk = 0; blk < p.bpt; ++blk) {
                    const int64_t e = x.first + x.t * p.bpt + blk;
                    int64_t id = e < x.end ? static_cast<int64_t>(p.table[e]) : -1;
                    if (id < 0 || id >= p.max_blocks) id = 0;  // a dummy box; never scored
                    const int64_t row = ((p.layer_slots + id) * p.nkv + x.c) * p.bs;
                    for (int kc = 0; kc < p.kchunks; ++kc) {
                        tma_load_2d(dst + kc * (kTileTokens * p.row_bytes) +
                                        blk * p.bs * p.row_bytes,
                                    &tmap_a, &a_full[stage], kc * elems_per_row,
                                    static_cast<int32_t>(row));
                    }
                }
                ++issued;
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                raise_error(p.dev_status, p.lib_error, HSS_ERR_DEVICE_TIMEOUT);
                *(volatile int*)abort_flag = 1;
            }
            // Drain: every copy this thread started has landed before the CTA may exit.
            const int64_t outstanding = issued < p.stages ? issued : p.stages;
            for (int64_t k = 1; k <= outstanding; ++k) {
                const int64_t n = issued - k;
                (void)mbar_wait(&a_full[n % p.stages], static_cast<uint32_t>((n / p.stages) & 1));
            }
            if (b_loads > 0) (void)mbar_wait(b_full, (b_loads - 1) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kTileTokens, kNChunk);
            int stage = 0;
            uint32_t phase = 0, b_full_phase = 0;
            int64_t prev_pair = -1, it = 0;
            bool ok = true;
            Unit x = first_unit;
            for (int64_t u = u_begin; u < u_end && ok;
                 ++u, advance_unit(x, p, units_before, offs)) {
                if (x.pair != prev_pair) {
                    if (prev_pair >= 0) umma_commit(b_empty);  // old slice free once MMAs finish
                    ok = mbar_wait(b_full, b_full_phase);
                    b_full_phase ^= 1u;
                    prev_pair = x.pair;
                    if (!ok) break;
                }
                if (!mbar_wait(&a_full[stage], phase) || *(volatile int*)abort_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // The descriptors' start-address field holds the byte address >> 4 (14 bits; the
                // shared-memory window stays below 256 KiB), so stepping through the operands
                // adds (offset >> 4) to a base descriptor: the single issuing thread spends a
                // few instructions per MMA, not a descriptor build (a chunk is only K = r deep).
                const uint64_t a_desc0 = smem_desc_kmajor(smem_u32(sA + stage * p.a_stage_bytes),
                                                          p.row_bytes);
                const uint64_t b_desc0 = smem_desc_kmajor(smem_u32(sB), p.row_bytes);
                const uint32_t a_kc = (kTileTokens * p.row_bytes) >> 4;
                const uint32_t b_kc = (p.slice * p.row_bytes) >> 4;
                const uint32_t b_nc = (kNChunk * p.row_bytes) >> 4;
                const int ksteps = elems_per_row / 16;
                for (int nc = 0; nc < nchunks && ok; ++nc, ++it) {
                    const int acc = static_cast<int>(it & 1);
                    if (!mbar_wait(&t_empty[acc], static_cast<uint32_t>(((it >> 1) & 1) ^ 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kNChunk);
                    uint64_t ad_kc = a_desc0, bd_kc = b_desc0 + nc * b_nc;
                    for (int kc = 0; kc < p.kchunks; ++kc, ad_kc += a_kc, bd_kc += b_kc) {
                        for (int ks = 0; ks < ksteps; ++ks) {
                            // ks * 32 bytes along K inside the swizzled rows: + 2 per step
                            umma_bf16(d_tmem, ad_kc + 2 * ks, bd_kc + 2 * ks, idesc,
                                      (kc | ks) != 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(&t_full[acc]);
                }
                umma_commit(&a_empty[stage]);
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                raise_error(p.dev_status, p.lib_error, HSS_ERR_DEVICE_TIMEOUT);
                *(volatile int*)abort_flag = 1;
            }
        }
    } else {
        // Epilogue: warpgroup eg drains columns [128 eg, 128 eg + 128) of every chunk; warp w
        // owns TMEM lanes 32 * (w % 4) .. + 31 = token rows of the tile.
        const int eg = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int token = quarter * 32 + lane;
        int64_t it = 0;  // global chunk counter, shared numbering with the MMA warp
        bool ok = true;
        // (masked mode and per-row mode with g <= 2: each unit decoded afresh, their
        // epilogues have no registers to spare)
        Unit x = first_unit;
        for (int64_t u = u_begin; u < u_end && ok; ++u) {
            if constexpr ((ROWG > 0 && ROWG < 4) || MASKED) {
                x = decode_unit(u, q_slice, p, units_before, offs);
            } else if (u > u_begin) {
                advance_unit(x, p, units_before, offs);
            }
            float run = -INFINITY;
            bool any = false;
            // This lane's block and whether its id is valid, looked up once per unit, before
            // the first chunk's wait (which hides the load).
            const int64_t blk_e = x.first + x.t * p.bpt + token / p.bs;
            const bool blk_in = blk_e < x.end;
            bool row_ok = false;
            if (blk_in) {
                const int64_t id = p.table[blk_e];
                row_ok = id >= 0 && id < p.max_blocks;
                if (!row_ok && x.c == 0 && x.q == 0 && (lane & (p.bs - 1)) == 0)
                    raise_error(p.dev_status, p.lib_error, HSS_ERR_OUT_OF_RANGE);
            }
            const int64_t row_st = x.end - x.first, row_ee = blk_e - x.first;
            // This thread's token position; with masks, the token may be hidden (past the
            // context) or visible only to query rows from some row on (causal).
            bool tok_ok = true;
            int64_t first_vec = 0;
            if (MASKED) {
                const int64_t tok_pos =
                    (x.t * p.bpt + token / p.bs) * static_cast<int64_t>(p.bs) + (token % p.bs);
                tok_ok = ctx_len == nullptr || tok_pos < __ldg(&ctx_len[x.s]);
                // First visible query vector: rows r >= tok_pos - row_pos0, i.e. vectors from
                // (tok_pos - row_pos0) * g on.
                first_vec = row_pos0 == nullptr ? 0 : (tok_pos - __ldg(&row_pos0[x.s])) * p.g;
            }
            for (int nc = 0; nc < nchunks; ++nc, ++it) {
                const int acc = static_cast<int>(it & 1);
                const bool got = mbar_wait(&t_full[acc], static_cast<uint32_t>((it >> 1) & 1));
                if (__any_sync(0xffffffffu, !got) || *(volatile int*)abort_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const int col0 = eg * 128;
                // Query vectors of this warpgroup's columns: v0 .. v0 + 127, valid below nvec.
                const int v0 = x.q * p.slice + nc * kNChunk + col0;
                const int valid = min(128, p.nvec - v0);
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(acc * kNChunk + col0);
                if constexpr (ROWG >= 4) {
                    // 128 / g <= 32 rows: the columns come in two halves of 64, each folded to
                    // row maxima at once; the accumulator is released before the shuffles.
                    constexpr int V = 128 / ROWG;
                    float xr[V];
                    if (valid == 128) {
                        // Every column real: each row's max over its g heads (g consecutive
                        // columns) is taken in the TMEM load path, one reduction per row.
#pragma unroll
                        for (int i = 0; i < V; ++i)
                            xr[i] = tmem_ldred_max<ROWG>(taddr + static_cast<uint32_t>(i * ROWG));
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < V; ++i) order_after_wait(xr[i]);
                    } else if (valid > 0) {
                        uint32_t va[64];
                        tmem_ld_32x32b_x32(taddr, va);
                        tmem_ld_32x32b_x32(taddr + 32, va + 32);
                        tmem_ld_wait();
                        group_max64<ROWG, 0>(va, valid, xr);
                        tmem_ld_32x32b_x32(taddr + 64, va);
                        tmem_ld_32x32b_x32(taddr + 96, va + 32);
                        tmem_ld_wait();
                        group_max64<ROWG, V / 2>(va, valid - 64, xr);
                    }
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&t_empty[acc]);
                    if (valid > 0) {
                        const bool e_ok = row_ok;
                        const int64_t st = row_st, ee = row_ee;
                        if (p.bs == 16)
                            scatter_rows<ROWG, 16>(xr, v0, lane, p.rows, p.scores, st, ee, e_ok);
                        else
                            scatter_rows<ROWG, 32>(xr, v0, lane, p.rows, p.scores, st, ee, e_ok);
                    }
                    continue;
                } else if constexpr (ROWG > 0) {
                    // g 1 or 2: all 128 columns to registers, the accumulator released, then
                    // 32 columns (32 / g rows) at a time.
                    uint32_t v[128];
                    if (valid > 0) {
                        tmem_ld_32x32b_x32(taddr, v);
                        tmem_ld_32x32b_x32(taddr + 32, v + 32);
                        tmem_ld_32x32b_x32(taddr + 64, v + 64);
                        tmem_ld_32x32b_x32(taddr + 96, v + 96);
                        tmem_ld_wait();
                    }
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&t_empty[acc]);
                    if (valid > 0) {
                        const bool e_ok = row_ok;
                        const int64_t st = row_st, ee = row_ee;
                        if (p.bs == 16) {
                            rows_to_scores<ROWG, 16, 0, 32>(v, valid, v0, lane, p.rows, p.scores, st, ee, e_ok);
                            if (valid > 32) rows_to_scores<ROWG, 16, 32, 32>(v, valid - 32, v0 + 32, lane, p.rows, p.scores, st, ee, e_ok);
                            if (valid > 64) rows_to_scores<ROWG, 16, 64, 32>(v, valid - 64, v0 + 64, lane, p.rows, p.scores, st, ee, e_ok);
                            if (valid > 96) rows_to_scores<ROWG, 16, 96, 32>(v, valid - 96, v0 + 96, lane, p.rows, p.scores, st, ee, e_ok);
                        } else {
                            rows_to_scores<ROWG, 32, 0, 32>(v, valid, v0, lane, p.rows, p.scores, st, ee, e_ok);
                            if (valid > 32) rows_to_scores<ROWG, 32, 32, 32>(v, valid - 32, v0 + 32, lane, p.rows, p.scores, st, ee, e_ok);
                            if (valid > 64) rows_to_scores<ROWG, 32, 64, 32>(v, valid - 64, v0 + 64, lane, p.rows, p.scores, st, ee, e_ok);
                            if (valid > 96) rows_to_scores<ROWG, 32, 96, 32>(v, valid - 96, v0 + 96, lane, p.rows, p.scores, st, ee, e_ok);
                        }
                    }
                    continue;
                } else if (!MASKED && valid == 128) {
                    // Every column a real query vector: the max over them is taken in the
                    // TMEM load path (four 32-column reductions), no register copy to scan.
                    any = true;
                    float m0 = tmem_ldred_max_x32(taddr);
                    float m1 = tmem_ldred_max_x32(taddr + 32);
                    float m2 = tmem_ldred_max_x32(taddr + 64);
                    float m3 = tmem_ldred_max_x32(taddr + 96);
                    tmem_ld_wait_values(m0, m1, m2, m3);
                    run = fmax3(run, fmaxf(m0, m1), fmaxf(m2, m3));
                } else if (valid > 0) {
                    any = true;
                    uint32_t v[128];
                    tmem_ld_32x32b_x32(taddr, v);
                    tmem_ld_32x32b_x32(taddr + 32, v + 32);
                    tmem_ld_32x32b_x32(taddr + 64, v + 64);
                    tmem_ld_32x32b_x32(taddr + 96, v + 96);
                    tmem_ld_wait();
                    int lo_col = 0;
                    if (MASKED) {
                        const int64_t lo64 = first_vec - v0;
                        lo_col = lo64 <= 0 ? 0 : (lo64 >= 128 ? 128 : static_cast<int>(lo64));
                    }
                    if (MASKED && (!tok_ok || lo_col >= valid)) {
                        // nothing visible in these columns
                    } else if (MASKED && lo_col > 0) {
#pragma unroll
                        for (int j = 0; j < 128; ++j)
                            if (j >= lo_col && j < valid) run = fmaxf(run, __uint_as_float(v[j]));
                    } else if (valid == 128) {
                        float m0 = run, m1 = run, m2 = run, m3 = run;
#pragma unroll
                        for (int j = 0; j < 128; j += 8) {
                            m0 = fmax3(m0, __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                            m1 = fmax3(m1, __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                            m2 = fmax3(m2, __uint_as_float(v[j + 4]), __uint_as_float(v[j + 5]));
                            m3 = fmax3(m3, __uint_as_float(v[j + 6]), __uint_as_float(v[j + 7]));
                        }
                        run = fmax3(fmaxf(m0, m1), m2, m3);
                    } else {
#pragma unroll
                        for (int j = 0; j < 128; ++j)
                            if (j < valid) run = fmaxf(run, __uint_as_float(v[j]));
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&t_empty[acc]);
            }
            if (!ok) break;
            if constexpr (ROWG > 0) continue;  // per-row scores went out chunk by chunk
            if (!any) continue;  // none of this warpgroup's columns held a valid query vector
            // Max over the block's tokens: block_size consecutive lanes.
            for (int off = p.bs >> 1; off > 0; off >>= 1)
                run = fmaxf(run, __shfl_xor_sync(0xffffffffu, run, off));
            if ((lane & (p.bs - 1)) == 0 && blk_in)
                atomic_max_f32(p.scores + blk_e, row_ok ? run : INFINITY);
        }
        if (!ok && lane == 0) {
            raise_error(p.dev_status, p.lib_error, HSS_ERR_DEVICE_TIMEOUT);
            *(volatile int*)abort_flag = 1;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

int g_smem_set[64] = {0};
std::mutex g_smem_mu;

}  // namespace

bool score_tc_supported(const ScoreArgs& a) {
    if (a.num_seqs < 1 || a.num_seqs > kMaxSeqs) return false;
    if (a.block_size != 16 && a.block_size != 32) return false;
    if (a.r % 16 != 0 || a.r < 16 || a.r > 256) return false;
    const int g = a.num_q_heads / a.num_kv_heads;
    if (g < 1 || g > kNChunk || kNChunk % g != 0) return false;
    if (a.r > 64 && a.r % 64 != 0) return false;
    const TcLayout L = make_tc_layout(a.r, 232448);
    return L.stages >= 2;
}

namespace {

using TcKernel = void (*)(CUtensorMap, CUtensorMap, TcParams, const int32_t*, const int32_t*,
                          int64_t);

TcKernel tc_kernel_for(bool masked, int rowg) {
    switch (rowg) {
        case 0: return masked ? score_tc_kernel<true, 0> : score_tc_kernel<false, 0>;
        case 1: return score_tc_kernel<false, 1>;
        case 2: return score_tc_kernel<false, 2>;
        case 4: return score_tc_kernel<false, 4>;
        case 8: return score_tc_kernel<false, 8>;
        case 16: return score_tc_kernel<false, 16>;
        default: return nullptr;
    }
}

// rowg == 0: block scores (scores [total]); rowg == g: per-row scores of one sequence
// (scores [rows_per_seq, total]).
hss_status launch_tc(const ScoreArgs& a, int rowg, cudaStream_t stream) {
    if (a.total == 0) return HSS_OK;
    const DeviceInfo* dev = current_device_info();
    if (dev == nullptr) return HSS_ERR_CUDA;
    if (!score_tc_supported(a)) return HSS_ERR_UNSUPPORTED_SHAPE;
    const bool masked = a.ctx_len != nullptr || a.row_pos0 != nullptr;
    const TcKernel kern = tc_kernel_for(masked, rowg);
    if (kern == nullptr || (rowg > 0 && (masked || a.num_seqs != 1))) return HSS_ERR_UNSUPPORTED_SHAPE;
    const TcLayout L = make_tc_layout(a.r, dev->max_smem_optin);
    if (L.stages < 2) return HSS_ERR_UNSUPPORTED_SHAPE;
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return HSS_ERR_CUDA;
    const int g = a.num_q_heads / a.num_kv_heads;
    const int elems = L.row_bytes / 2;
    const CUtensorMapSwizzle sw = L.row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : L.row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_32B;
    // A_g as rows of r: row ((layer * max_blocks + id) * nkv + c) * bs + t.  The map spans
    // every layer up to the scored one, so rows of the scored layer are in range.
    CUtensorMap tmap_a, tmap_q;
    {
        const uint64_t rows = static_cast<uint64_t>(a.layer_offset_slots + a.max_blocks) *
                              a.num_kv_heads * a.block_size;
        const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(a.r), rows};
        const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(a.r) * 2};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(elems),
                                   static_cast<cuuint32_t>(a.block_size)};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&tmap_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.A_g), gdim,
                gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return HSS_ERR_CUDA;
    }
    {
        // Qp as [num_seqs * rows][num_q_heads][r]; a box is 256 query vectors of one kv
        // head: (256 / g) rows x g heads x one swizzled row segment.
        const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(a.r),
                                    static_cast<cuuint64_t>(a.num_q_heads),
                                    static_cast<cuuint64_t>(a.num_seqs) * a.rows_per_seq};
        const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(a.r) * 2,
                                       static_cast<cuuint64_t>(a.num_q_heads) * a.r * 2};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(elems), static_cast<cuuint32_t>(g),
                                   static_cast<cuuint32_t>(kNChunk / g)};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.Qp), gdim,
                gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return HSS_ERR_CUDA;
    }
    {
        std::lock_guard<std::mutex> lk(g_smem_mu);
        const int d = dev->device & 63;
        if (g_smem_set[d] < L.total_bytes) {
            const TcKernel all[] = {score_tc_kernel<false, 0>, score_tc_kernel<true, 0>,
                                    score_tc_kernel<false, 1>, score_tc_kernel<false, 2>,
                                    score_tc_kernel<false, 4>, score_tc_kernel<false, 8>,
                                    score_tc_kernel<false, 16>};
            for (TcKernel k : all)
                if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L.total_bytes) != cudaSuccess)
                    return HSS_ERR_CUDA;
            g_smem_set[d] = L.total_bytes;
        }
    }
    TcParams p;
    p.table = a.table;
    p.seq_offsets = a.seq_offsets;
    p.scores = a.scores;
    p.dev_status = a.dev_status;
    p.lib_error = dev->error_word;
    p.layer_slots = a.layer_offset_slots;
    p.max_blocks = a.max_blocks;
    p.num_seqs = a.num_seqs;
    p.nkv = a.num_kv_heads;
    p.g = g;
    p.bs = a.block_size;
    p.r = a.r;
    p.rows = a.rows_per_seq;
    p.nvec = a.rows_per_seq * g;
    p.slice = std::min(L.slice, (p.nvec + kNChunk - 1) / kNChunk * kNChunk);
    p.b_bytes = p.slice * a.r * 2;
    p.nslices = (p.nvec + p.slice - 1) / p.slice;
    p.bpt = kTileTokens / a.block_size;
    p.row_bytes = L.row_bytes;
    p.kchunks = L.kchunks;
    p.a_stage_bytes = L.a_stage_bytes;
    p.stages = L.stages;
    // Units per slice: exact for one sequence; otherwise an upper bound (the offsets live on
    // the device), since every sequence contributes ceil(n_s / bpt) <= n_s / bpt + 1 tiles.
    const int64_t max_tiles = a.num_seqs == 1 ? (a.total + p.bpt - 1) / p.bpt
                                              : a.total / p.bpt + a.num_seqs;
    const int64_t units = static_cast<int64_t>(p.nkv) * max_tiles;
    // One CTA per SM, in groups of nslices (one CTA per slice).
    int64_t groups = std::max<int64_t>(1, dev->num_sms / p.nslices);
    groups = std::min<int64_t>(groups, units);
    p.num_groups = static_cast<int32_t>(groups);
    p.units_per_group = (units + groups - 1) / groups;
    const int grid = static_cast<int>(groups * p.nslices);

    float* scores = a.scores;
    const int64_t total = rowg > 0 ? a.total * a.rows_per_seq : a.total;
    const int fill_grid = static_cast<int>(std::min<int64_t>((total + 255) / 256, 1024));
    if (launch_pdl(fill_neg_inf, dim3(fill_grid), dim3(256), 0, stream, scores, total) !=
        cudaSuccess)
        return HSS_ERR_CUDA;
    const int64_t one_total = a.total;
    if (launch_pdl(kern, dim3(grid), dim3(kThreads), L.total_bytes, stream, tmap_a, tmap_q, p,
                   a.ctx_len, a.row_pos0, one_total) != cudaSuccess)
        return HSS_ERR_CUDA;
    return HSS_OK;
}

}  // namespace

hss_status launch_score_tc(const ScoreArgs& a, cudaStream_t stream) {
    return launch_tc(a, 0, stream);
}

hss_status launch_score_tc_rows(const ScoreArgs& a, cudaStream_t stream) {
    return launch_tc(a, a.num_q_heads / a.num_kv_heads, stream);
}

}  // namespace hss
