// score_decode_kernel.cuh -- the decode scorer's kernel and its per-shape launchers.
// Included by score_decode.cu (the host dispatcher, which only declares the launchers'
// instances) and by score_decode_k{1,2,4,8}.cu, each of which instantiates the kernels of one
// r = 16 * KSTEPS, so that the build compiles them in parallel.
//
// Block scores in the decode regime (few query vectors per kv head).
//
// Page "metrale_storage/predictor.rs", Predictor::score_blocks: each block's score is the max,
// over query heads and the block's tokens, of the projected dot product Qp . A_g, where query
// head h reads kv head h / g.  Here a block table and several query rows per sequence are
// added; an identity table reproduces the page's contiguous slots.
//
// The regime is HBM-bound: each block's A_g slot (num_kv_heads * block_size * r bf16, 8 KiB
// for the Llama-3-8B-like layer) is read exactly once, and only ~2 FMAs are done per byte.
// Design:
//   * one warp scores one block at a time; a warp owns a contiguous run of table entries;
//   * the slot is read with 16-byte coalesced loads straight into registers -- all of a
//     block's loads are issued before any arithmetic, so each warp keeps up to 8 KiB in flight;
//   * the arithmetic runs on the warp-level tensor-core MMA (m16n8k16, bf16 in, fp32
//     accumulate): tokens are the M side (16 per tile), the query vectors of one kv group
//     (rows x g heads) the N side, r the K side.  Because the score only needs the dot product
//     over r, the r-coordinates may be visited in any order as long as A and B use the same
//     one; the order is chosen so that each lane's 16-byte load *is* its A fragment;
//   * the query-vector fragments of the current sequence sit in a per-warp shared-memory
//     cache in fragment order (one 8-byte load per MMA);
//   * the max over tokens and query vectors is reduced in registers, then across the warp
//     with shuffles; padded query-vector columns are masked to -inf.
#pragma once

#include <algorithm>
#include <atomic>
#include <cmath>
#include <type_traits>

#include "rank_device.cuh"

namespace hss {
namespace decode {

constexpr int kWarpsMax = 8;
constexpr int kFragBudgetBytes = 48 * 1024;  // per CTA, all warps' fragment caches
// In-kernel query projection: at most this many sequences per call (every CTA projects all of
// them) and this much shared memory for their fragment caches, P's fragments and Q's rows.
constexpr int kInlineMaxSeqs = 8;
constexpr int kInlineBudgetBytes = 96 * 1024;

struct DecodeParams {
    const uint16_t* Qp;
    const uint16_t* A_g;
    const int32_t* table;
    const int32_t* seq_offsets;
    float* scores;
    int32_t* dev_status;
    int32_t* lib_error;
    int64_t layer_slots;
    int64_t max_blocks;
    int64_t total;
    int64_t entries_per_warp;
    int32_t num_seqs;
    int32_t rows;
    int32_t nq;
    int32_t nkv;
    int32_t r;
    int32_t bs;
    int32_t g;
    int32_t nvec;  // rows * g query vectors per kv head
    // Fused victim ranking (counters == nullptr: off).  counters[s] counts the entries of
    // sequence s scored so far; the CTA that completes a sequence ranks it and resets the
    // counter to zero.
    int32_t* counters;
    int32_t* victims;
    int32_t k;
    int32_t sel_cap;
    int32_t frag_bytes_cta;  // offset of the ranking scratch in shared memory
    int32_t todo_cap;        // sequences one CTA can complete: its entry count
    // early != 0: the previous kernel in the stream writes only Qp and the A_g slots listed
    // in new_ids, so the rest may be read before the grid dependency wait.
    const int32_t* new_ids;
    int32_t num_new;
    int32_t early;
    // Optional masks (nullptr = off): token position p = j * bs + t for the entry at table
    // position j of its sequence; p < ctx_len[s]; causal: p <= row_pos0[s] + row.
    const int32_t* ctx_len;
    const int32_t* row_pos0;
    // INLINE kernels project the queries themselves (Qp is never stored): every CTA projects
    // Q [num_seqs, rows, nq, hd] through P [hd, r] straight into a shared-memory cache of
    // MMA B fragments, one per sequence.  Shared memory: that cache (cache_bytes), P's
    // fragments (r * hd * 2 bytes), then Q's rows (row stride hd + 32 elements).
    const uint16_t* Q;
    const uint16_t* P;
    int32_t hd;
    int32_t cache_bytes;
    // nowait != 0 (INLINE only): the previous kernel in the stream is this call's projection
    // of the new_ids slots and nothing else, so only a warp about to read one of those slots
    // takes the grid dependency wait; num_new <= 32 then.
    int32_t nowait;
    // spread != 0 (one sequence of at most kSpreadMaxEntries entries, every CTA of the grid
    // resident at once, 8-byte aligned workspace): instead of the last CTA ranking the whole
    // sequence, every CTA publishes its entries' keys as call-tagged words, waits until every
    // word of the sequence carries this call's tag and places its own entries by counting the
    // smaller words, so the ranking is spread over the grid.
    int32_t spread;
    // TMA kernels (INLINE, at most 2 entries per warp, slots of at most 8 KiB): each warp's
    // slots arrive by one bulk copy per entry into its shared-memory buffer, completion counted
    // on the warp's mbarrier, instead of through the warp's own loads.  Offsets of the eight
    // mbarriers and of the eight slot buffers in shared memory.
    int32_t tma_bar_off;
    int32_t tma_buf_off;
    // Spread ranking's wait on the other CTAs' words: its limit, and (self-test only, else -1)
    // a CTA that withholds its words so that every other CTA's wait runs out.
    uint64_t wait_limit_ns;
    int32_t withhold_cta;
};

// TMA slot buffers: the largest slot and the most entries per warp they take.
constexpr int kTmaMaxSlotBytes = 8192;
constexpr int kTmaMaxEntriesPerWarp = 2;

// Spread ranking: keys per thread (256 threads) and so the longest sequence it takes.
constexpr int kSpreadKeysPerThread = 16;
constexpr int kSpreadMaxEntries = kWarpsMax * 32 * kSpreadKeysPerThread;
// ... and the most entries one CTA scores and places (2 per warp at 4096 entries on 152 SMs).
constexpr int kSpreadMaxCta = 16;
// Its workspace region (p.counters in spread mode): the call number (a line of its own), then
// from byte 256 one tagged word per entry (32 KiB).
constexpr int kSpreadWordsOffsetWords = 64;
// ... at most this many sequences (their index takes 3 bits of a word), and the call number's
// bits kept in a word (above the sequence and the 32-bit key).
constexpr int kSpreadMaxSeqs = 8;
constexpr uint32_t kSpreadTagMask = (1u << 29) - 1u;

// below -= [w < we] for 64-bit unsigned words: one borrow chain, no predicate or branch (a
// compare-and-select per pair issued about twice the instructions).
__device__ __forceinline__ void sub_if_less(uint32_t& below, uint64_t w, uint64_t we) {
    asm("{\n\t"
        ".reg .u32 t;\n\t"
        "sub.cc.u32 t, %1, %3;\n\t"
        "subc.cc.u32 t, %2, %4;\n\t"
        "subc.u32 %0, %0, 0;\n\t"
        "}"
        : "+r"(below)
        : "r"(static_cast<uint32_t>(w)), "r"(static_cast<uint32_t>(w >> 32)),
          "r"(static_cast<uint32_t>(we)), "r"(static_cast<uint32_t>(we >> 32)));
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t* addr) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u64(uint64_t* addr, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu_s32(int* addr, int v) {
    asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// Totals over the warp of eight per-lane counts: afterwards lane l holds the total of
// c[(l >> 2) & 7].  Three exchanges each halve the counts a lane carries (it keeps the half
// its lane bit selects and adds its partner's copy of that half), then two plain ones finish
// the sums: nine shuffles for eight totals.
__device__ __forceinline__ uint32_t warp_sum8(const uint32_t (&c)[8]) {
    const int lane = static_cast<int>(threadIdx.x) & 31;
    const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
    uint32_t a[4], h[2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        a[i] = (b4 ? c[i + 4] : c[i]) + __shfl_xor_sync(0xffffffffu, b4 ? c[i] : c[i + 4], 16);
#pragma unroll
    for (int i = 0; i < 2; ++i)
        h[i] = (b3 ? a[i + 2] : a[i]) + __shfl_xor_sync(0xffffffffu, b3 ? a[i] : a[i + 2], 8);
    uint32_t x = (b2 ? h[1] : h[0]) + __shfl_xor_sync(0xffffffffu, b2 ? h[0] : h[1], 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
}

// Spread ranking's gather: polls the call's n published words (slot q of thread t holds
// position t + 256 q) until each carries the tag, and in every round counts the words that
// arrived in it below each of the CTA's entries' counting words: neg[u] -= that count.  A
// slot in which no lane of the warp saw a word arrive is skipped, so the counting mostly
// overlaps the wait for the last CTA's words.  Returns false when the wait ran out.
template <int SLOTS, int E>
__device__ __forceinline__ bool spread_gather_count(const uint64_t* words, int n, uint32_t tag,
                                                    const uint64_t (&we)[E], uint32_t (&neg)[E],
                                                    uint64_t limit_ns) {
    uint32_t missing = 0;
#pragma unroll
    for (int q = 0; q < SLOTS; ++q)
        if (static_cast<int>(threadIdx.x) + q * kWarpsMax * 32 < n) missing |= 1u << q;
    const uint64_t t0 = global_timer_ns();
    while (__any_sync(0xffffffffu, missing != 0)) {
        uint64_t v[SLOTS];
#pragma unroll
        for (int q = 0; q < SLOTS; ++q) {
            const int j = static_cast<int>(threadIdx.x) + q * kWarpsMax * 32;
            v[q] = (missing >> q) & 1u ? ld_relaxed_gpu_u64(&words[j]) : 0ull;
        }
        uint32_t arrived = 0;
#pragma unroll
        for (int q = 0; q < SLOTS; ++q) {
            const int j = static_cast<int>(threadIdx.x) + q * kWarpsMax * 32;
            const bool now = ((missing >> q) & 1u) && static_cast<uint32_t>(v[q] >> 35) == tag;
            arrived |= static_cast<uint32_t>(now) << q;
            // the counting word: sequence << 44 | key << 12 | position
            v[q] = now ? (((v[q] >> 32) & 7ull) << 44) | ((v[q] & 0xFFFFFFFFull) << 12) |
                             static_cast<uint32_t>(j)
                       : ~0ull;
        }
        missing &= ~arrived;
#pragma unroll
        for (int q = 0; q < SLOTS; ++q)
            if (__any_sync(0xffffffffu, (arrived >> q) & 1u))
#pragma unroll
                for (int u = 0; u < E; ++u) sub_if_less(neg[u], v[q], we[u]);
        if (__any_sync(0xffffffffu, missing != 0 && global_timer_ns() - t0 > limit_ns))
            return false;
    }
    return true;
}

// The CTA's cnt <= E entries (positions pos0 .. pos0 + cnt - 1 of the call, keys keys[],
// sequences from the S + 1 offsets soff relative to the call's first entry eb - pos0): gathers
// every word, counts those below each entry's word and leaves this warp's count of entry e in
// part_warp[e].  Returns false when the wait ran out.
template <int E>
__device__ __forceinline__ bool spread_count(const uint64_t* words, int n, uint32_t tag,
                                             uint64_t limit_ns, const int32_t* soff, int S,
                                             const uint32_t* keys, int64_t eb, int pos0,
                                             int cnt, uint32_t* part_warp) {
    uint64_t we[E];
    uint32_t neg[E];
#pragma unroll
    for (int u = 0; u < E; ++u) {
        int se = 0;  // entry u's sequence
        for (int t = 1; t < S; ++t) se += static_cast<int64_t>(soff[t]) <= eb + u;
        we[u] = u < cnt ? (static_cast<uint64_t>(se) << 44) |
                              (static_cast<uint64_t>(keys[u]) << 12) |
                              static_cast<uint32_t>(pos0 + u)
                        : 0ull;  // no word lies below it
        neg[u] = 0;
    }
    const bool ok = n <= 8 * kWarpsMax * 32
                        ? spread_gather_count<8, E>(words, n, tag, we, neg, limit_ns)
                        : spread_gather_count<16, E>(words, n, tag, we, neg, limit_ns);
    const int lane = static_cast<int>(threadIdx.x) & 31;
#pragma unroll
    for (int g = 0; g < E / 8; ++g) {
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = neg[8 * g + i];
        const uint32_t tot = 0u - warp_sum8(c);
        const int e = 8 * g + ((lane >> 2) & 7);
        if ((lane & 3) == 0 && e < cnt) part_warp[e] = tot;
    }
    return ok;
}

__device__ __forceinline__ int atom_add_acq_rel_gpu(int* addr, int v) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Physical r-offset of the 4 elements that lane quad t holds for k-step ks
// (KSTEPS even: each 16-byte load covers two k-steps; KSTEPS == 1: 8-byte loads).
template <int KSTEPS>
__device__ __forceinline__ int frag_r_offset(int ks, int t) {
    if constexpr (KSTEPS == 1) {
        return 4 * t;
    } else {
        return 32 * (ks >> 1) + 8 * t + 4 * (ks & 1);
    }
}

// MASKED: the call passed ctx_len or row_pos0.  A template parameter, so the unmasked kernel
// carries none of the mask arithmetic.  INLINE: the queries are projected in the kernel.
// TMA: slots arrive by bulk copies into shared memory (INLINE kernels only).
template <int KSTEPS, int NT, bool MASKED, bool INLINE, bool TMA>
__global__ void __launch_bounds__(kWarpsMax * 32, 2) score_decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(16) uint8_t smem_dec[];
    uint2* frag_cache_all = reinterpret_cast<uint2*>(smem_dec);
    constexpr int kLoadsPerRow = KSTEPS == 1 ? 1 : KSTEPS / 2;  // 16-byte (or 8-byte) loads
    constexpr int kRegsPerTile = KSTEPS == 1 ? 4 : 4 * KSTEPS;  // both row halves
    constexpr int kTilesPerBatch = 64 / kRegsPerTile;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2;  // MMA group id: token row (A), query vector column (B)
    const int tq = lane & 3;   // thread in group
    const int frag_per_warp = p.nkv * KSTEPS * NT * 32;
    uint2* cache = frag_cache_all + warp * frag_per_warp;

    const int64_t wid = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
    const int64_t i_begin = wid * p.entries_per_warp;
    const bool has_work = i_begin < p.total;
    const int64_t i_end = min(p.total, i_begin + p.entries_per_warp);

    const int tiles_per_head = p.bs >> 4;
    const int num_tiles = p.nkv * tiles_per_head;
    const int64_t slot_elems = static_cast<int64_t>(p.nkv) * p.bs * p.r;
    const int64_t tile_elems = 16 * static_cast<int64_t>(p.r);

    // One batch of a slot's 16-token tiles, straight into MMA A-fragment registers, from
    // global memory (streaming loads) or from the slot's copy in shared memory (TMA kernels;
    // the same layout).
    uint32_t data[kTilesPerBatch][kRegsPerTile];
    auto issue_loads_from = [&](const uint16_t* slot, int tb, auto in_smem) {
        constexpr bool kSmem = decltype(in_smem)::value;
#pragma unroll
        for (int u = 0; u < kTilesPerBatch; ++u) {
            const int tile = tb + u;
            if (tile < num_tiles) {
                const uint16_t* base = slot + tile * tile_elems;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint16_t* rowp = base + (gq + 8 * half) * p.r;
#pragma unroll
                    for (int l = 0; l < kLoadsPerRow; ++l) {
                        if constexpr (KSTEPS == 1) {
                            const uint2* src = reinterpret_cast<const uint2*>(rowp + 4 * tq);
                            const uint2 v = kSmem ? *src : __ldcs(src);
                            data[u][half * 2 + 0] = v.x;
                            data[u][half * 2 + 1] = v.y;
                        } else {
                            const uint4* src = reinterpret_cast<const uint4*>(rowp + 32 * l + 8 * tq);
                            const uint4 v = kSmem ? *src : __ldcs(src);
                            data[u][(half * kLoadsPerRow + l) * 4 + 0] = v.x;
                            data[u][(half * kLoadsPerRow + l) * 4 + 1] = v.y;
                            data[u][(half * kLoadsPerRow + l) * 4 + 2] = v.z;
                            data[u][(half * kLoadsPerRow + l) * 4 + 3] = v.w;
                        }
                    }
                }
            }
        }
    };
    auto issue_loads = [&](const uint16_t* slot, int tb) {
        issue_loads_from(slot, tb, std::false_type{});
    };
    // TMA kernels: the warp's slot buffer and its mbarrier.  A slot's copy is started by lane 0
    // (expect the bytes, then one bulk copy); the warp waits on the barrier's current phase
    // before it reads the buffer.  Issuing 8 KiB of per-lane loads per warp kept the SM's load
    // queue busy for ~1 us, and every shared-memory access issued after them waited behind
    // them; the bulk copies bypass that queue.
    uint64_t* tma_bar = reinterpret_cast<uint64_t*>(smem_dec + p.tma_bar_off) + warp;
    uint16_t* tma_buf = reinterpret_cast<uint16_t*>(smem_dec + p.tma_buf_off) + warp * slot_elems;
    uint32_t tma_parity = 0;
    const uint32_t slot_bytes = static_cast<uint32_t>(slot_elems * 2);
    auto tma_start = [&](int32_t id) {
        if (lane == 0) {
            mbar_arrive_expect_tx(tma_bar, slot_bytes);
            bulk_copy_g2s(tma_buf, p.A_g + (p.layer_slots + id) * slot_elems, slot_bytes, tma_bar);
        }
    };
    // Issue a slot's data: loads into the registers, or (TMA) the bulk copy.
    auto start_slot = [&](int32_t id) {
        if constexpr (TMA)
            tma_start(id);
        else
            issue_loads(p.A_g + (p.layer_slots + id) * slot_elems, 0);
    };
    if constexpr (TMA) {
        if (lane == 0) mbar_init(tma_bar, 1);
        fence_mbarrier_init();
        __syncwarp();
    }
    // The last s with seq_offsets[s] <= i, searched 32 ways at a time: each round the lanes
    // load 32 evenly spaced offsets of the range at once (one L2 round trip for up to 32
    // sequences, two for up to 1024).  Whole warp.
    auto find_seq = [&](int64_t i) {
        int lo = 0, hi = p.num_seqs;  // seq_offsets[lo] <= i; the answer is below hi
        while (hi - lo > 1) {
            const int step = (hi - lo + 31) >> 5;
            const int j = lo + lane * step;
            const bool le = j < hi && static_cast<int64_t>(__ldg(&p.seq_offsets[j])) <= i;
            const unsigned below = __ballot_sync(0xffffffffu, le);  // a prefix of the lanes
            lo += (31 - __clz(below)) * step;
            hi = min(hi, lo + step);
        }
        return lo;
    };

    int s = 0;
    int64_t seq_end = 0;
    int32_t my_id = 0;
    bool have_ids = false;  // my_id already holds the first batch's entries
    bool preloaded = false;
    // INLINE: the staging loads (Q's rows by asynchronous copies, P's first two pieces per
    // thread into registers) are requested before any slot data: Q of a layer is touched once
    // per model step and comes from DRAM, where it queued behind the 16 MiB of slot traffic
    // (~3 us) when it was requested after it.
    uint4* pfrag = reinterpret_cast<uint4*>(smem_dec + p.cache_bytes);
    uint16_t* pfrag_h = reinterpret_cast<uint16_t*>(pfrag);
    uint16_t* qs = reinterpret_cast<uint16_t*>(smem_dec + p.cache_bytes + p.r * p.hd * 2);
    const int qstride = p.hd + 32;  // padded rows: conflict-free fragment reads
    const int qvec = p.hd >> 3;
    const int pvec = p.r >> 3;  // 16-byte pieces per row of P: 2, 4, 8 or 16
    const int pshift = __ffs(pvec) - 1;
    const int p_items = p.hd * pvec;
    uint4 pv[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
    bool staged = false;
    auto stage_issue = [&]() {
        for (int z = threadIdx.x; z < p.cache_bytes / 16; z += blockDim.x)
            reinterpret_cast<uint4*>(smem_dec)[z] = make_uint4(0u, 0u, 0u, 0u);
        const int M = p.rows * p.nq;
        for (int e = threadIdx.x; e < p.num_seqs * M * qvec; e += blockDim.x) {
            const int row = e / qvec, c8 = e - row * qvec;
            cp_async_16(qs + row * qstride + 8 * c8, p.Q + static_cast<int64_t>(row) * p.hd + 8 * c8);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = static_cast<int>(threadIdx.x) + u * static_cast<int>(blockDim.x);
            const int dd = e >> pshift, jc = e & (pvec - 1);
            if (e < p_items) pv[u] = __ldg(reinterpret_cast<const uint4*>(p.P + dd * p.r) + jc);
        }
        staged = true;
    };
    // Spread ranking: the call's offsets and its number (the word the previous call advanced)
    // are copied into shared memory before any slot is requested (behind the slots' traffic
    // their round trip took microseconds), by asynchronous copies that hold no registers;
    // they are waited for with the queries' rows, or before this CTA's keys go out.
    bool spread_issued = false;
    auto spread_issue = [&]() {
        spread_issued = true;
        if (!p.spread) return;
        uint32_t* tag_smem = reinterpret_cast<uint32_t*>(smem_dec + p.frag_bytes_cta) + p.todo_cap +
                             kWarpsMax * kSpreadMaxCta;
        if (static_cast<int>(threadIdx.x) <= p.num_seqs)
            cp_async_4(tag_smem + 4 + threadIdx.x, p.seq_offsets + threadIdx.x);
        if (threadIdx.x == 0) cp_async_16(tag_smem, p.counters);  // L2 only: the current word
    };
    if (INLINE && p.early) {
        stage_issue();  // the previous kernel writes neither Q nor P
        spread_issue();
    }

    if (p.early && has_work) {
        // The previous kernel in the stream is this call's own projection, which writes only
        // Qp and the slots of new_ids: the offsets, the table and every other slot may be
        // read before the dependency wait, so the first block's DRAM latency overlaps it.
        const int64_t first_n = i_end - i_begin < 32 ? i_end - i_begin : 32;
        my_id = lane < first_n ? __ldg(&p.table[i_begin + lane]) : 0;
        have_ids = true;
        // num_new <= 64: two new ids per lane, loaded alongside the table entries.
        const int32_t nid0 = lane < p.num_new ? __ldg(&p.new_ids[lane]) : -1;
        const int32_t nid1 = lane + 32 < p.num_new ? __ldg(&p.new_ids[lane + 32]) : -1;
        s = find_seq(i_begin);
        seq_end = __ldg(&p.seq_offsets[s + 1]);
        const int32_t id0 = __shfl_sync(0xffffffffu, my_id, 0);
        const bool fresh = __any_sync(0xffffffffu, nid0 == id0 || nid1 == id0);
        if (id0 >= 0 && id0 < p.max_blocks && !fresh) {
            start_slot(id0);
            preloaded = true;
        }
    }
    const bool nowait = INLINE && p.nowait != 0;
    if (!nowait) grid_dependency_wait();
    // Spread ranking waits for every CTA of this grid: the next kernel is let in only once a
    // CTA has published its keys (all CTAs are then resident, so it cannot take their places).
    if (!p.spread) grid_launch_dependents();
    // nowait: this lane's new id (lane < num_new <= 32); a warp waits before its first one.
    const int32_t my_new = nowait && lane < p.num_new ? __ldg(&p.new_ids[lane]) : -1;
    bool waited = !nowait;
    if (!spread_issued) spread_issue();

    if constexpr (INLINE) {
        if (!staged) stage_issue();
        // The first block's loads go out before the projection below, so their DRAM latency
        // covers it (without this call's own projection before the scorer they could not be
        // issued before the dependency wait).
        if (has_work && !preloaded) {
            const int64_t first_n = i_end - i_begin < 32 ? i_end - i_begin : 32;
            my_id = lane < first_n ? __ldg(&p.table[i_begin + lane]) : 0;
            have_ids = true;
            s = find_seq(i_begin);
            seq_end = __ldg(&p.seq_offsets[s + 1]);
            const int32_t id0 = __shfl_sync(0xffffffffu, my_id, 0);
            if (id0 >= 0 && id0 < p.max_blocks && !__any_sync(0xffffffffu, my_new == id0)) {
                start_slot(id0);
                preloaded = true;
            }
        }
        // ---- project every sequence's queries into the CTA's fragment cache
        // P goes to shared memory as MMA B fragments.  The head_dim coordinates are visited in
        // the order that makes each lane's 16-byte load of a query row its A fragment for two
        // k-steps (the scheme the slot loads use for r), so B takes the same order: fragment
        // entry (n-tile np, 32-wide chunk l, lane) holds P[32l + 8t + e][8np + g] as its e-th
        // bf16 (t = lane % 4, g = lane / 4).  Pieces past the first two per thread are loaded
        // two at a time here.
        const int lchunks = p.hd >> 5;
        const int M = p.rows * p.nq;
        auto scatter_p = [&](const uint4 (&v)[2], int e0) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int e = e0 + u * static_cast<int>(blockDim.x);
                if (e < p_items) {
                    const int dd = e >> pshift, jc = e & (pvec - 1);
                    const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                    const int base =
                        ((jc * lchunks + (dd >> 5)) * 32 + ((dd & 31) >> 3)) * 8 + (dd & 7);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)  // column 8 jc + jj sits in lane group jj
                        pfrag_h[base + jj * 32] =
                            static_cast<uint16_t>(w[jj >> 1] >> ((jj & 1) * 16));
                }
            }
        };
        scatter_p(pv, static_cast<int>(threadIdx.x));
        for (int e0 = static_cast<int>(threadIdx.x) + 2 * static_cast<int>(blockDim.x);
             e0 < p_items; e0 += 2 * static_cast<int>(blockDim.x)) {
            uint4 v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int e = e0 + u * static_cast<int>(blockDim.x);
                const int dd = e >> pshift, jc = e & (pvec - 1);
                v[u] = e < p_items ? __ldg(reinterpret_cast<const uint4*>(p.P + dd * p.r) + jc)
                                   : make_uint4(0u, 0u, 0u, 0u);
            }
            scatter_p(v, e0);
        }
        cp_async_wait_all();
        __syncthreads();
        // Tasks: (sequence, 16 query vectors m, 8 columns j of r).  Vector m = row * nq + h
        // (Q's own row order); D[m][j] = sum_d Q[m][d] P[d][j] in fp32, rounded to bf16 once,
        // then stored where the scoring loop expects Qp[v][j] of kv head h / g, v = row * g +
        // h % g: fragment (c, k-step, n-tile v / 8), lane (v % 8) * 4 + t, word half h2, with
        // (k-step, t, h2) the inverse of frag_r_offset.
        const int mtiles = (M + 15) >> 4;
        const int ntp = p.r >> 3;
        const int ntask = p.num_seqs * mtiles * ntp;
        uint32_t* cache_words = reinterpret_cast<uint32_t*>(smem_dec);
        for (int task = warp; task < ntask; task += static_cast<int>(blockDim.x >> 5)) {
            const int np = task % ntp;
            const int mt = (task / ntp) % mtiles;
            const int sq = task / (ntp * mtiles);
            const int m0 = 16 * mt + gq, m1 = m0 + 8;
            const uint16_t* q0 = qs + (sq * M + m0) * qstride + 8 * tq;
            const uint16_t* q1 = q0 + 8 * qstride;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            for (int l = 0; l < lchunks; ++l) {
                const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
                const uint4 x0 = m0 < M ? *reinterpret_cast<const uint4*>(q0 + 32 * l) : zero;
                const uint4 x1 = m1 < M ? *reinterpret_cast<const uint4*>(q1 + 32 * l) : zero;
                const uint4 b = pfrag[(np * lchunks + l) * 32 + lane];
                mma_bf16_16816(d, x0.x, x1.x, x0.y, x1.y, b.x, b.y);
                mma_bf16_16816(d, x0.z, x1.z, x0.w, x1.w, b.z, b.w);
            }
            const int j0 = 8 * np + 2 * tq;  // this lane's columns j0, j0 + 1
            int ks, t2;
            if constexpr (KSTEPS == 1) {
                ks = 0;
                t2 = j0 >> 2;
            } else {
                ks = 2 * (j0 >> 5) + ((j0 & 7) >> 2);
                t2 = (j0 & 31) >> 3;
            }
            const int h2 = (j0 & 3) >> 1;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int m = hh ? m1 : m0;
                if (m < M) {
                    const int row = m / p.nq;
                    const int h = m - row * p.nq;
                    const int c = h / p.g;
                    const int v = row * p.g + (h - c * p.g);
                    const int frag = ((sq * p.nkv + c) * KSTEPS + ks) * NT + (v >> 3);
                    cache_words[(frag * 32 + (v & 7) * 4 + t2) * 2 + h2] =
                        pack_bf16x2(d[2 * hh], d[2 * hh + 1]);
                }
            }
        }
        __syncthreads();
    }
    if (has_work) {
    if (!p.early) {
        s = find_seq(i_begin);
        seq_end = __ldg(&p.seq_offsets[s + 1]);
    }
    int cached_seq = -1;
    // Spread ranking: each entry's key goes to shared memory as it is scored.
    uint32_t* spread_key = reinterpret_cast<uint32_t*>(smem_dec + p.frag_bytes_cta);
    const int64_t spread_first =
        static_cast<int64_t>(blockIdx.x) * p.entries_per_warp * (blockDim.x >> 5);
    int64_t seq_begin = MASKED ? __ldg(&p.seq_offsets[s]) : 0;
    int64_t clen = INT64_MAX, pos0 = INT64_MAX / 2;
    if (MASKED) {
        if (p.ctx_len != nullptr) clen = __ldg(&p.ctx_len[s]);
        if (p.row_pos0 != nullptr) pos0 = __ldg(&p.row_pos0[s]);
    }

    // Column validity of this lane's accumulator entries (query vector index < nvec).
    // Masked kernels: the query row of each of those entries (vector / g), computed once.
    bool col_ok[NT][2];
    int col_row[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            col_ok[nt][cc] = nt * 8 + 2 * tq + cc < p.nvec;
            col_row[nt][cc] = MASKED ? (nt * 8 + 2 * tq + cc) / p.g : 0;
        }
    }

    for (int64_t i0 = i_begin; i0 < i_end; i0 += 32) {
        const int64_t left = i_end - i0;
        const int n_here = left < 32 ? static_cast<int>(left) : 32;
        if (!(have_ids && i0 == i_begin)) my_id = lane < n_here ? __ldg(&p.table[i0 + lane]) : 0;
        for (int e = 0; e < n_here; ++e) {
            const int64_t i = i0 + e;
            while (i >= seq_end && s + 1 < p.num_seqs) {
                ++s;
                seq_end = __ldg(&p.seq_offsets[s + 1]);
                if (MASKED) {
                    seq_begin = __ldg(&p.seq_offsets[s]);
                    if (p.ctx_len != nullptr) clen = __ldg(&p.ctx_len[s]);
                    if (p.row_pos0 != nullptr) pos0 = __ldg(&p.row_pos0[s]);
                }
            }
            const int32_t id = __shfl_sync(0xffffffffu, my_id, e);
            if (id < 0 || id >= p.max_blocks) {
                if (lane == 0) {
                    p.scores[i] = INFINITY;
                    if (p.spread) spread_key[i - spread_first] = rankdev::rank_key<false>(INFINITY);
                    raise_error(p.dev_status, p.lib_error, HSS_ERR_OUT_OF_RANGE);
                }
                continue;
            }
            if (!waited && __any_sync(0xffffffffu, my_new == id)) {
                grid_dependency_wait();  // the slot is being written by the previous kernel
                waited = true;
            }
            const uint16_t* slot = p.A_g + (p.layer_slots + id) * slot_elems;
            if constexpr (TMA) {
                // The buffer holds one slot: the previous entry's reads are done (and ordered
                // before the async proxy's writes) before the next copy starts.
                if (!(preloaded && i == i_begin)) {
                    __syncwarp();
                    fence_proxy_async_smem();
                    tma_start(id);
                }
                if (!mbar_wait(tma_bar, tma_parity)) {
                    // Bounded: a copy that has not landed in 1 s is reported, not waited for.
                    if (lane == 0) raise_error(p.dev_status, p.lib_error, HSS_ERR_DEVICE_TIMEOUT);
                }
                tma_parity ^= 1u;
                slot = tma_buf;
            }
            float best = -INFINITY;
            for (int tb = 0; tb < num_tiles; tb += kTilesPerBatch) {
                // Issue every load of the batch first (the first one may already be in flight).
                if constexpr (TMA)
                    issue_loads_from(slot, tb, std::true_type{});
                else if (!(preloaded && i == i_begin && tb == 0))
                    issue_loads(slot, tb);
                // (Re)fill the query-vector fragment cache while the loads are in flight.
                if (INLINE && s != cached_seq) {
                    cache = frag_cache_all + s * frag_per_warp;  // the CTA's projection
                    cached_seq = s;
                } else if (s != cached_seq) {
                    // Fragment (c, ks, nt) is entry (c * KSTEPS + ks) * NT + nt; 8 per lane are
                    // loaded before any is stored, so the refill costs one L2 round trip per
                    // 8 fragments (not one per kv head).
                    constexpr int kBatch = 8;
                    const int nfrag = p.nkv * KSTEPS * NT;
                    __syncwarp();
                    for (int f0 = 0; f0 < nfrag; f0 += kBatch) {
                        uint2 f[kBatch];
#pragma unroll
                        for (int u = 0; u < kBatch; ++u) {
                            const int fi = f0 + u;
                            const int nt = fi % NT, ks = (fi / NT) % KSTEPS;
                            const int c = fi / (NT * KSTEPS);
                            const int v = nt * 8 + gq;
                            f[u] = make_uint2(0u, 0u);
                            if (fi < nfrag && v < p.nvec) {
                                const int row = v / p.g;
                                const int h = c * p.g + (v - row * p.g);
                                const uint16_t* q =
                                    p.Qp + ((static_cast<int64_t>(s) * p.rows + row) * p.nq + h) *
                                               p.r;
                                f[u] = *reinterpret_cast<const uint2*>(
                                    q + frag_r_offset<KSTEPS>(ks, tq));
                            }
                        }
#pragma unroll
                        for (int u = 0; u < kBatch; ++u)
                            if (f0 + u < nfrag) cache[(f0 + u) * 32 + lane] = f[u];
                    }
                    __syncwarp();
                    cached_seq = s;
                }
                // One 16-token tile: the MMAs over r for kv head c, then the max into `best`.
                auto score_tile = [&](const int u, const int c, const int in_head) {
                    float acc[NT][4];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
                    for (int ks = 0; ks < KSTEPS; ++ks) {
                        uint32_t a0, a1, a2, a3;
                        if constexpr (KSTEPS == 1) {
                            a0 = data[u][0];  // token row gq,     r 4t..4t+1
                            a2 = data[u][1];  // token row gq,     r 4t+2..4t+3
                            a1 = data[u][2];  // token row gq + 8
                            a3 = data[u][3];
                        } else {
                            const int l = ks >> 1, w = ks & 1;
                            a0 = data[u][(0 * kLoadsPerRow + l) * 4 + 2 * w + 0];
                            a2 = data[u][(0 * kLoadsPerRow + l) * 4 + 2 * w + 1];
                            a1 = data[u][(1 * kLoadsPerRow + l) * 4 + 2 * w + 0];
                            a3 = data[u][(1 * kLoadsPerRow + l) * 4 + 2 * w + 1];
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 b = cache[((c * KSTEPS + ks) * NT + nt) * 32 + lane];
                            mma_bf16_16816(acc[nt], a0, a1, a2, a3, b.x, b.y);
                        }
                    }
                    if (!MASKED) {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            best = fmaxf(best, col_ok[nt][0] ? fmaxf(acc[nt][0], acc[nt][2])
                                                             : -INFINITY);
                            best = fmaxf(best, col_ok[nt][1] ? fmaxf(acc[nt][1], acc[nt][3])
                                                             : -INFINITY);
                        }
                    } else {
                        // Accumulator rows are tokens gq and gq + 8 of this 16-token tile,
                        // columns are query vectors (row = vector / g).
                        const int64_t p_lo = (i - seq_begin) * p.bs + in_head * 16 + gq;
                        const int64_t p_hi = p_lo + 8;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                            for (int cc = 0; cc < 2; ++cc) {
                                if (!col_ok[nt][cc]) continue;
                                const int64_t lim = min(clen - 1, pos0 + col_row[nt][cc]);
                                if (p_lo <= lim) best = fmaxf(best, acc[nt][cc]);
                                if (p_hi <= lim) best = fmaxf(best, acc[nt][cc + 2]);
                            }
                        }
                    }
                };
                // kv head c of the batch's first tile and the tile's place in its head, then
                // stepped tile by tile with selects.  A division, or a branch around each tile,
                // in the unrolled bodies below would serialise them: each tile's fragment
                // loads and MMAs would wait for the one before (measured: 5x the arithmetic
                // time of a block).  Only a batch that runs past the last tile tests each tile.
                int c = 0, in_head = 0;
                if (tb != 0) {
                    c = tb / tiles_per_head;
                    in_head = tb - c * tiles_per_head;
                }
                if (tb + kTilesPerBatch <= num_tiles) {
#pragma unroll
                    for (int u = 0; u < kTilesPerBatch; ++u) {
                        score_tile(u, c, in_head);
                        const bool wrap = in_head + 1 == tiles_per_head;
                        in_head = wrap ? 0 : in_head + 1;
                        c += wrap ? 1 : 0;
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < kTilesPerBatch; ++u) {
                        if (tb + u < num_tiles) score_tile(u, c, in_head);
                        const bool wrap = in_head + 1 == tiles_per_head;
                        in_head = wrap ? 0 : in_head + 1;
                        c += wrap ? 1 : 0;
                    }
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, off));
            if (lane == 0) {
                p.scores[i] = best;
                if (p.spread) spread_key[i - spread_first] = rankdev::rank_key<false>(best);
            }
        }
    }
    }  // has_work
    if (p.counters == nullptr) return;

    if (p.spread) {
        // ---- spread ranking of the call's S <= 8 sequences, at most 4096 entries in all.
        // Every CTA publishes its entries' keys in the workspace as 64-bit words tagged with
        // this call's number (tag << 35 | sequence << 32 | key, one relaxed store each) and
        // reads all the call's words until every one carries the tag: each word is its own
        // completion flag, so no counter, fence or second read of the scores is needed.
        // The rank of entry e of sequence s is then the number of counting words
        // (sequence << 44 | key << 12 | position) below its own, less the entries of the
        // sequences before s (their words all lie below); entry e is victim number rank(e)
        // of its sequence when that is below k.  The words are unique, so within a sequence
        // the ranks are a permutation, ordered by (key, position).
        uint32_t* ekey = reinterpret_cast<uint32_t*>(smem_dec + p.frag_bytes_cta);
        uint32_t* part = ekey + p.todo_cap;  // [warp][kSpreadMaxCta] partial counts, then
        uint32_t* tag_smem = part + kWarpsMax * kSpreadMaxCta;  // the last call's number,
        int32_t* soff = reinterpret_cast<int32_t*>(tag_smem + 4);  // seq_offsets[0 .. S],
        uint8_t* eseq = reinterpret_cast<uint8_t*>(soff + kSpreadMaxSeqs + 1);  // entries' seqs
        const int S = p.num_seqs;
        const int64_t per_cta = p.entries_per_warp * (blockDim.x >> 5);
        const int64_t cb = static_cast<int64_t>(blockIdx.x) * per_cta;
        int* epoch = p.counters;
        uint64_t* words = reinterpret_cast<uint64_t*>(p.counters + kSpreadWordsOffsetWords);
        cp_async_wait_all();  // the offsets and the call number
        __syncthreads();  // this CTA's keys, the call number and the offsets
        const int64_t a = soff[0], b = soff[S];
        if (a < 0 || b < a || b > p.total || b - a > kSpreadMaxEntries) {
            // Offsets that do not describe at most 4096 of the scored entries: nothing is
            // published (the keys region holds 4096 words).
            if (threadIdx.x == 0) raise_error(p.dev_status, p.lib_error, HSS_ERR_OUT_OF_RANGE);
            grid_launch_dependents();
            return;
        }
        const int n = static_cast<int>(b - a);
        const int64_t eb = max(cb, a), ee = min(min(p.total, cb + per_cta), b);
        const int cnt = ee > eb ? static_cast<int>(ee - eb) : 0;  // <= kSpreadMaxCta
        // Sequences with fewer entries than k end their rows with -1 (CTA 0 writes them).
        auto pad_rows = [&]() {
            if (blockIdx.x != 0) return;
            for (int q = 0; q < S; ++q) {
                const int nq = soff[q + 1] - soff[q];
                for (int j = max(nq, 0) + static_cast<int>(threadIdx.x); j < p.k; j += blockDim.x)
                    p.victims[static_cast<int64_t>(q) * p.k + j] = -1;
            }
        };
        if (cnt == 0) {  // no entry of the call in this CTA
            pad_rows();
            grid_launch_dependents();
            return;
        }
        const uint32_t tag = (*tag_smem + 1u) & kSpreadTagMask;  // this call's number
        const int pos0 = static_cast<int>(eb - a);  // position of this CTA's first entry
        // (self-test: the withheld CTA, an index past the grid meaning its last one)
        const int withheld = p.withhold_cta < 0 ? -1
                             : min(p.withhold_cta, static_cast<int>(gridDim.x) - 1);
        if (static_cast<int>(threadIdx.x) < cnt) {
            const int64_t i = eb + threadIdx.x;
            int se = 0;  // this entry's sequence
            while (se + 1 < S && soff[se + 1] <= i) ++se;
            eseq[threadIdx.x] = static_cast<uint8_t>(se);
            if (static_cast<int>(blockIdx.x) != withheld)
                st_relaxed_gpu_u64(&words[pos0 + threadIdx.x],
                                   (static_cast<uint64_t>(tag) << 35) |
                                       (static_cast<uint64_t>(se) << 32) | ekey[eb - cb + threadIdx.x]);
        }
        // Every CTA that gets here is resident and has published (or holds no entry): the next
        // kernel may take free places now; it cannot take ours.
        grid_launch_dependents();
        // Gather every word, counting as they arrive; each warp leaves its count of each of
        // the CTA's entries in `part` (no atomics).
        const bool ok = cnt <= 8
            ? spread_count<8>(words, n, tag, p.wait_limit_ns, soff, S, ekey + (eb - cb), eb,
                              pos0, cnt, part + warp * kSpreadMaxCta)
            : spread_count<16>(words, n, tag, p.wait_limit_ns, soff, S, ekey + (eb - cb), eb,
                               pos0, cnt, part + warp * kSpreadMaxCta);
        if (!ok && lane == 0) raise_error(p.dev_status, p.lib_error, HSS_ERR_DEVICE_TIMEOUT);
        __syncthreads();  // every thread has seen every word; the counts and eseq are set
        // Every CTA has published, so every CTA has read the tag: the CTA holding the call's
        // first entry advances the call number for the next call.
        if (threadIdx.x == 0 && static_cast<int64_t>(blockIdx.x) == a / per_cta)
            st_relaxed_gpu_s32(epoch, static_cast<int>(tag));
        if (static_cast<int>(threadIdx.x) < cnt) {
            const int se = eseq[threadIdx.x];
            uint32_t below = 0;
#pragma unroll
            for (int wv = 0; wv < kWarpsMax; ++wv) below += part[wv * kSpreadMaxCta + threadIdx.x];
            const int64_t first = soff[se];  // the words of earlier sequences all lie below
            const uint32_t rank = below - static_cast<uint32_t>(first - a);
            if (rank < static_cast<uint32_t>(p.k))
                p.victims[static_cast<int64_t>(se) * p.k + rank] =
                    static_cast<int32_t>(eb + threadIdx.x - first);
        }
        pad_rows();
        return;
    }

    // ---- fused ranking: the CTA that completes a sequence ranks it
    constexpr int kThreadsFused = kWarpsMax * 32;
    uint8_t* rank_smem = smem_dec + p.frag_bytes_cta;
    uint64_t* sel = reinterpret_cast<uint64_t*>(rank_smem);
    rankdev::RankShared* sh = reinterpret_cast<rankdev::RankShared*>(sel + p.sel_cap);
    int* todo = reinterpret_cast<int*>(sh + 1);  // [todo_cap + 1]
    // The barrier orders every warp's scores before thread 0's count, which is a release at
    // GPU scope (cumulative over what the barrier made visible to it); the count of the CTA
    // that completes a sequence is also an acquire, so that CTA sees every other CTA's scores.
    __syncthreads();
    if (threadIdx.x == 0) {
        int ntodo = 0;
        const int64_t per_cta = p.entries_per_warp * (blockDim.x >> 5);
        const int64_t cb = static_cast<int64_t>(blockIdx.x) * per_cta;
        const int64_t ce = min(p.total, cb + per_cta);
        if (cb < ce) {
            int lo2 = 0, hi2 = p.num_seqs;  // last s with seq_offsets[s] <= cb
            while (hi2 - lo2 > 1) {
                const int mid = (lo2 + hi2) >> 1;
                if (static_cast<int64_t>(__ldg(&p.seq_offsets[mid])) <= cb) lo2 = mid; else hi2 = mid;
            }
            for (int q = lo2; q < p.num_seqs; ++q) {
                const int64_t a = __ldg(&p.seq_offsets[q]), b = __ldg(&p.seq_offsets[q + 1]);
                if (a >= ce) break;
                const int64_t cnt = min(ce, b) - max(cb, a);
                if (cnt <= 0) continue;
                const int old = atom_add_acq_rel_gpu(&p.counters[q], static_cast<int>(cnt));
                if (old + cnt == b - a && ntodo < p.todo_cap) todo[1 + ntodo++] = q;
            }
        }
        todo[0] = ntodo;
    }
    __syncthreads();
    const int ntodo = todo[0];
    for (int t = 0; t < ntodo; ++t) {
        const int q = todo[1 + t];
        const int64_t a = __ldg(&p.seq_offsets[q]);
        const int n = static_cast<int>(__ldg(&p.seq_offsets[q + 1]) - a);
        rankdev::rank_sequence<kThreadsFused>(p.scores + a, n, p.k,
                                              p.victims + static_cast<int64_t>(q) * p.k, sel,
                                              p.sel_cap, sh);
        if (threadIdx.x == 0) p.counters[q] = 0;  // ready for the next call
    }
    // Empty sequences have no entries to complete them: CTA 0 writes their -1 rows.
    if (blockIdx.x == 0) {
        for (int q = threadIdx.x; q < p.num_seqs; q += blockDim.x) {
            if (__ldg(&p.seq_offsets[q + 1]) == __ldg(&p.seq_offsets[q])) {
                for (int j = 0; j < p.k; ++j) p.victims[static_cast<int64_t>(q) * p.k + j] = -1;
            }
        }
    }
}

template <int KSTEPS, int NT>
auto kernel_for(const DecodeParams& p) {
    const bool masked = p.ctx_len != nullptr || p.row_pos0 != nullptr;
    return p.Q != nullptr && p.tma_buf_off != 0 ? score_decode_kernel<KSTEPS, NT, false, true, true>
           : p.Q != nullptr ? score_decode_kernel<KSTEPS, NT, false, true, false>
           : masked         ? score_decode_kernel<KSTEPS, NT, true, false, false>
                            : score_decode_kernel<KSTEPS, NT, false, false, false>;
}

// CTAs of 256 threads with `smem` bytes of dynamic shared memory that one SM holds at once,
// for the kernel `p` selects (cached per kernel: the last shared-memory size asked for).
template <int KSTEPS, int NT>
int ctas_per_sm_t(const DecodeParams& p, int smem) {
    static std::atomic<uint64_t> cache[4];  // (smem << 32 | ctas) per kernel of kernel_for
    const int which = p.Q != nullptr ? (p.tma_buf_off != 0 ? 3 : 0)
                      : (p.ctx_len != nullptr || p.row_pos0 != nullptr) ? 1 : 2;
    const uint64_t c = cache[which].load(std::memory_order_relaxed);
    if (c != 0 && static_cast<int>(c >> 32) == smem) return static_cast<int>(c & 0xFFFFFFFFu);
    auto k = kernel_for<KSTEPS, NT>(p);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 0;
    int ctas = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas, k, kWarpsMax * 32, smem) !=
        cudaSuccess)
        return 0;
    cache[which].store((static_cast<uint64_t>(smem) << 32) | static_cast<uint32_t>(ctas),
                       std::memory_order_relaxed);
    return ctas;
}

template <int KSTEPS, int NT>
hss_status launch_t(const DecodeParams& p, int warps_per_cta, int smem, int grid,
                    cudaStream_t stream) {
    auto k = kernel_for<KSTEPS, NT>(p);
    if (smem > 48 * 1024) {
        // The largest dynamic shared memory already allowed, per kernel of kernel_for and
        // device: the attribute call is made only when a launch needs more (a host-side
        // saving on every layer call).
        static std::atomic<int> allowed[4][64];
        const int which = p.Q != nullptr ? (p.tma_buf_off != 0 ? 3 : 0)
                          : (p.ctx_len != nullptr || p.row_pos0 != nullptr) ? 1 : 2;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return HSS_ERR_CUDA;
        if (allowed[which][dev].load(std::memory_order_relaxed) < smem) {
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess)
                return HSS_ERR_CUDA;
            allowed[which][dev].store(smem, std::memory_order_relaxed);
        }
    }
    if (launch_pdl(k, dim3(grid), dim3(warps_per_cta * 32), smem, stream, p) != cudaSuccess)
        return HSS_ERR_CUDA;
    return HSS_OK;
}

}  // namespace decode
}  // namespace hss

// Explicit instances of the launchers (and through them the kernels) for r = 16 * KS: one
// translation unit defines them, the dispatcher only declares them.
#define HSS_DECODE_INSTANCES(PREFIX, KS)                                                    \
    PREFIX template int hss::decode::ctas_per_sm_t<KS, 1>(const hss::decode::DecodeParams&,  \
                                                          int);                              \
    PREFIX template int hss::decode::ctas_per_sm_t<KS, 2>(const hss::decode::DecodeParams&,  \
                                                          int);                              \
    PREFIX template hss_status hss::decode::launch_t<KS, 1>(const hss::decode::DecodeParams&, \
                                                            int, int, int, cudaStream_t);    \
    PREFIX template hss_status hss::decode::launch_t<KS, 2>(const hss::decode::DecodeParams&, \
                                                            int, int, int, cudaStream_t);
