// project_tc.cu -- Q and K projection, Y = bf16(X . P), on the 5th-generation tensor cores.
//
// Page "metrale_storage/predictor.rs": Predictor::project_q (q_proj = q @ P, stored BF16) and
// Predictor::project_kv_block (k_block [block_size, num_kv_heads, head_dim] projected into the
// head-major A_g slot [num_kv_heads, block_size, r], stored BF16).  Both are the same skinny
// GEMM -- rows of head_dim against P [head_dim, r] -- and differ only in where a result row
// is stored, so one kernel serves both.
//
// Design (persistent, warp-specialised, one CTA per SM):
//   warp 0      TMA producer: 128-row tiles of X, swizzled 128B, into a ring of smem stages
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma M=128, N=r, K=16 steps, fp32
//               accumulators double-buffered in TMEM (2 x r columns)
//   warps 2..5  epilogue: tcgen05.ld a row per thread, round to bf16, store the row
//   warps 6..9  cache copy (token/slot mode with a cache only): each tile's key rows, already
//               in shared memory, go to their slots in the paged key cache; the stage is free
//               once the MMAs and all four copy warps are done with it (no barrier among the
//               copy warps: each arrives on its own, so a wait that runs out cannot strand one)
// P^T stays resident in shared memory (K-major, 128B swizzle) for the whole kernel.
// The work is HBM-bound (head_dim * 2 bytes in, r * 2 bytes out per row); the tensor
// cores only keep the arithmetic far below the memory time.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "ptx.cuh"

namespace hss {
namespace {

constexpr int kBM = 128;            // rows per tile = UMMA M
constexpr int kChunkElems = 64;     // bf16 elements per 128-byte swizzled row segment
constexpr int kChunkBytes = kBM * 128;
constexpr int kThreads = 320;  // producer, MMA, 4 epilogue warps, 4 cache-copy warps
constexpr int kMaxStages = 6;

struct ProjLayout {
    int kchunks = 0;       // head_dim / 64
    int b_bytes = 0;       // P^T: kchunks * r * 128
    int stage_bytes = 0;   // kchunks * 128 rows * 128 B
    int stages = 0;
    int bar_offset = 0;    // from the 1024-aligned base
    int total_bytes = 0;   // dynamic smem to request (includes alignment slack)
    int tmem_cols = 0;
};

__host__ __device__ inline int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p <<= 1;
    return p;
}

__host__ __device__ inline ProjLayout make_layout(int head_dim, int r, int smem_budget) {
    ProjLayout L;
    L.kchunks = head_dim / kChunkElems;
    L.b_bytes = L.kchunks * r * 128;
    L.stage_bytes = L.kchunks * kChunkBytes;
    const int fixed = 1024 /*align slack*/ + 256 /*barriers*/ + L.b_bytes;
    int st = (smem_budget - fixed) / L.stage_bytes;
    L.stages = st < kMaxStages ? st : kMaxStages;
    L.bar_offset = L.b_bytes + L.stages * L.stage_bytes;
    L.total_bytes = 1024 + L.bar_offset + 256;
    L.tmem_cols = pow2_at_least(2 * r);
    return L;
}

// One launch projects up to two row segments (e.g. the query rows and the newly written
// key blocks of a decode step), each with its own input map and output mapping.
struct ProjSegment {
    int64_t num_rows;
    int64_t tiles;             // ceil(num_rows / 128)
    uint16_t* out;
    const int32_t* block_ids;  // whole blocks -> A_g slot rows
    const int64_t* slots;      // single tokens -> A_g rows (both null: rows go to out + m * r)
    uint16_t* cache;           // slots mode: the key row is also copied to cache[slot][h]
    const uint16_t* X;         // the input rows (for that copy)
};

struct ProjParams {
    const uint16_t* P;
    int32_t head_dim;
    int32_t r;
    ProjSegment seg[2];
    int32_t num_kv_heads;
    int32_t block_size;
    int64_t max_blocks;
    int64_t layer_slots;  // layer * max_blocks
    int32_t* dev_status;
    int32_t* lib_error;
};

__global__ void __launch_bounds__(kThreads, 2)
    project_kernel(const __grid_constant__ CUtensorMap tmap_x0,
                   const __grid_constant__ CUtensorMap tmap_x1, const ProjParams p,
                   const int stages) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const ProjLayout L = make_layout(p.head_dim, p.r, 0x7FFFFFFF);  // sizes only
    const int kchunks = L.kchunks;
    const int stage_bytes = L.stage_bytes;
    const int b_bytes = L.b_bytes;
    uint8_t* sB = smem;
    uint8_t* sA = smem + b_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sA + stages * stage_bytes);
    uint64_t* empty = full + stages;
    uint64_t* tfull = empty + stages;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = p.r;
    const int64_t num_tiles = p.seg[0].tiles + p.seg[1].tiles;

    if (threadIdx.x == 0) {
        const bool copy = p.seg[0].cache != nullptr || p.seg[1].cache != nullptr;
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], copy ? 5 : 1);  // the MMAs' commit (+ each copy warp)
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, L.tmem_cols);
        tmem_relinquish();
    }
    // Everything above is set-up that may overlap the previous kernel in the stream; global
    // memory is touched only after the dependency wait.
    tc_fence_before_sync();
    __syncthreads();  // barriers initialised, TMEM allocated
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp != 0) {
        // Warps 1..5 stage P^T while warp 0 already streams the first tiles in.  P^T goes
        // into shared memory K-major with the 128-byte swizzle the MMA descriptor names:
        // row j of chunk c holds P[64c .. 64c+63][j].  P is read with 16-byte loads, a batch
        // of four per thread in flight at once, then scattered into the transposed layout.
        constexpr int kStagers = kThreads - 32;
        const int t = static_cast<int>(threadIdx.x) - 32;
        const int n16 = p.head_dim * r / 8;  // 16-byte chunks of P (8 consecutive j each)
        const uint4* P16 = reinterpret_cast<const uint4*>(p.P);
        for (int base = t; base < n16; base += 4 * kStagers) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = base + u * kStagers;
                if (e < n16) v[u] = __ldg(&P16[e]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = base + u * kStagers;
                if (e >= n16) continue;
                const int d = (e * 8) / r, j0 = (e * 8) - d * r;
                const int c = d / kChunkElems, kk = d - c * kChunkElems;
                uint8_t* chunk = sB + c * r * 128;
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint16_t h = static_cast<uint16_t>(w[q >> 1] >> (16 * (q & 1)));
                    *reinterpret_cast<uint16_t*>(chunk + swizzled_offset(j0 + q, kk * 2, 128)) = h;
                }
            }
        }
        fence_proxy_async_smem();  // the generic-proxy P^T writes, visible to the tensor cores
        // Named barrier 1 joins warps 1..5 only: the MMA warp starts once P^T is complete.
        asm volatile("bar.sync 1, %0;" ::"n"(kThreads - 32) : "memory");
    }

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmap_x0);
            if (p.seg[1].tiles > 0) tma_prefetch_desc(&tmap_x1);
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                if (!mbar_wait(&empty[stage], phase ^ 1u) || *(volatile int*)abort_flag) {
                    raise_error(p.dev_status, p.lib_error, HSS_ERR_DEVICE_TIMEOUT);
                    *(volatile int*)abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(stage_bytes));
                uint8_t* dst = sA + stage * stage_bytes;
                const bool second = tile >= p.seg[0].tiles;
                const CUtensorMap* map = second ? &tmap_x1 : &tmap_x0;
                const int64_t local = second ? tile - p.seg[0].tiles : tile;
                for (int c = 0; c < kchunks; ++c) {
                    tma_load_2d(dst + c * kChunkBytes, map, &full[stage], c * kChunkElems,
                                static_cast<int32_t>(local * kBM));
                }
                ++issued;
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // Drain: every load this thread issued has landed before the CTA may exit.
            const int64_t outstanding = issued < stages ? issued : stages;
            for (int64_t q = 1; q <= outstanding; ++q) {
                const int64_t n = issued - q;  // load number n used stage n % stages
                const int st = static_cast<int>(n % stages);
                const uint32_t ph = static_cast<uint32_t>((n / stages) & 1);
                (void)mbar_wait(&full[st], ph);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, static_cast<uint32_t>(r));
            int stage = 0;
            uint32_t phase = 0;
            int64_t it = 0;
            for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
                const int acc = static_cast<int>(it & 1);
                const uint32_t acc_phase = static_cast<uint32_t>((it >> 1) & 1);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u) || !mbar_wait(&full[stage], phase) ||
                    *(volatile int*)abort_flag) {
                    raise_error(p.dev_status, p.lib_error, HSS_ERR_DEVICE_TIMEOUT);
                    *(volatile int*)abort_flag = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * r);
                // Descriptors step by (offset >> 4) from a base (the start-address field holds
                // the address >> 4 and never carries below 256 KiB).
                uint64_t ad = smem_desc_kmajor(smem_u32(sA + stage * stage_bytes), 128);
                uint64_t bd = smem_desc_kmajor(smem_u32(sB), 128);
                for (int c = 0; c < kchunks; ++c, ad += kChunkBytes >> 4, bd += (r * 128) >> 4) {
#pragma unroll
                    for (int s = 0; s < kChunkElems / 16; ++s)  // 32 bytes along K per step
                        umma_bf16(d_tmem, ad + 2 * s, bd + 2 * s, idesc, (c | s) != 0 ? 1u : 0u);
                }
                umma_commit(&empty[stage]);  // smem stage free once these MMAs have read it
                umma_commit(&tfull[acc]);    // accumulator ready for the epilogue
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp >= 6) {
        // Cache copy: warp 6 + w takes rows 32w .. 32w + 31 of each tile, read from the
        // swizzled stage and written to K_cache[slot][h].
        const bool copy = p.seg[0].cache != nullptr || p.seg[1].cache != nullptr;
        if (copy) {
            const int cw = warp - 6;
            const int row_bytes = p.head_dim * 2;
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                const bool ok = mbar_wait(&full[stage], phase);
                if (__any_sync(0xffffffffu, !ok) || *(volatile int*)abort_flag) {
                    if (lane == 0) {
                        raise_error(p.dev_status, p.lib_error, HSS_ERR_DEVICE_TIMEOUT);
                        *(volatile int*)abort_flag = 1;
                    }
                    break;
                }
                const bool second = tile >= p.seg[0].tiles;
                const ProjSegment& sg = second ? p.seg[1] : p.seg[0];
                const int64_t local = second ? tile - p.seg[0].tiles : tile;
                if (sg.cache != nullptr) {
                    // This warp's 32 rows: every lane looks up one row's destination at once,
                    // then the rows go out two at a time (16 lanes x 16 bytes per row piece).
                    const uint8_t* src = sA + stage * stage_bytes;
                    const int my_rr = cw * 32 + lane;
                    const int64_t my_m = local * kBM + my_rr;
                    int64_t my_dst = -1;  // element offset of the row in the cache, or -1
                    if (my_m < sg.num_rows) {
                        const int64_t i = my_m / p.num_kv_heads;
                        const int64_t h = my_m - i * p.num_kv_heads;
                        const int64_t sl = sg.slots[i];
                        if (sl >= 0 && sl < p.max_blocks * p.block_size)
                            my_dst = (sl * p.num_kv_heads + h) * p.head_dim;
                    }
                    for (int k = 0; k < 16; ++k) {
                        const int pick = 2 * k + (lane >> 4);
                        const int64_t dst = __shfl_sync(0xffffffffu, my_dst, pick);
                        const int rr = cw * 32 + pick;
                        if (dst < 0) continue;
                        uint8_t* drow = reinterpret_cast<uint8_t*>(sg.cache + dst);
                        for (int cb = (lane & 15) * 16; cb < row_bytes; cb += 256) {
                            const int kc = cb >> 7, c16 = (cb & 127) >> 4;
                            const uint4 val = *reinterpret_cast<const uint4*>(
                                src + kc * kChunkBytes + rr * 128 + ((c16 ^ (rr & 7)) << 4));
                            *reinterpret_cast<uint4*>(drow + cb) = val;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);  // this warp is done with the stage
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        // Epilogue: warp w reads TMEM lanes 32 * (w % 4) .. + 31, one output row per thread.
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        const int rows_per_block = p.block_size * p.num_kv_heads;
        int64_t it = 0;
        for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
            const int acc = static_cast<int>(it & 1);
            const uint32_t acc_phase = static_cast<uint32_t>((it >> 1) & 1);
            // The row's slot or block id is requested before the wait for the accumulator, so
            // the lookup's latency overlaps it; the destination is formed after.
            const bool second = tile >= p.seg[0].tiles;
            const ProjSegment& sg = second ? p.seg[1] : p.seg[0];
            const int64_t m = (second ? tile - p.seg[0].tiles : tile) * kBM + row_in_tile;
            const bool have = m < sg.num_rows;
            int64_t look = -1;  // the token's slot, or the block's id
            int h = 0, t = 0, rem = 0;
            if (have) {
                if (sg.slots != nullptr) {
                    // Row m = (token i, kv head h); the token's slot names block and position.
                    const int64_t i = m / p.num_kv_heads;
                    h = static_cast<int>(m - i * p.num_kv_heads);
                    look = sg.slots[i];
                } else if (sg.block_ids != nullptr) {
                    const int64_t i = m / rows_per_block;
                    rem = static_cast<int>(m - i * rows_per_block);
                    t = rem / p.num_kv_heads;
                    h = rem - t * p.num_kv_heads;
                    look = sg.block_ids[i];
                }
            }
            const bool ok = mbar_wait(&tfull[acc], acc_phase);
            if (__any_sync(0xffffffffu, !ok) || *(volatile int*)abort_flag) {
                if (lane == 0) {
                    raise_error(p.dev_status, p.lib_error, HSS_ERR_DEVICE_TIMEOUT);
                    *(volatile int*)abort_flag = 1;
                }
                break;
            }
            tc_fence_after_sync();
            uint16_t* dst = nullptr;
            if (have) {
                if (sg.slots != nullptr) {
                    const int64_t sl = look;
                    if (sl >= 0 && sl < p.max_blocks * p.block_size) {
                        const int64_t blk = sl / p.block_size;
                        const int tt = static_cast<int>(sl - blk * p.block_size);
                        dst = sg.out + (((p.layer_slots + blk) * p.num_kv_heads + h) *
                                            p.block_size + tt) * static_cast<int64_t>(r);
                    } else if (sl >= 0 && h == 0) {
                        raise_error(p.dev_status, p.lib_error, HSS_ERR_OUT_OF_RANGE);
                    }
                } else if (sg.block_ids == nullptr) {
                    dst = sg.out + m * r;
                } else {
                    const int64_t id = look;
                    if (id >= 0 && id < p.max_blocks) {
                        dst = sg.out + (((p.layer_slots + id) * p.num_kv_heads + h) * p.block_size +
                                       t) * static_cast<int64_t>(r);
                    } else if (rem == 0) {
                        raise_error(p.dev_status, p.lib_error, HSS_ERR_OUT_OF_RANGE);
                    }
                }
            }
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * r);
            for (int c0 = 0; c0 < r; c0 += 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(taddr + c0, v);
                tmem_ld_wait();
                if (dst != nullptr) {
                    uint4 o0, o1;
                    o0.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
                    o0.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
                    o0.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
                    o0.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
                    o1.x = pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9]));
                    o1.y = pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11]));
                    o1.z = pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13]));
                    o1.w = pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15]));
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
                    d4[0] = o0;
                    d4[1] = o1;
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, L.tmem_cols);
    }
}

// ------------------------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    });
    return g_encode;
}

// The smem attribute is set once per device (value = the largest request so far).
int g_smem_set[64] = {0};
std::mutex g_smem_mu;

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return encoder(); }

bool project_shape_supported(int32_t head_dim, int32_t r) {
    if (head_dim <= 0 || head_dim % kChunkElems != 0 || head_dim > 256) return false;
    if (r < 16 || r > 256 || r % 16 != 0) return false;
    const ProjLayout L = make_layout(head_dim, r, 232448);
    return L.stages >= 2;
}

static bool encode_rows_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map,
                            const uint16_t* X, int64_t rows, int32_t head_dim) {
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(head_dim) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kChunkElems), static_cast<cuuint32_t>(kBM)};
    const cuuint32_t estride[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(X), gdim, gstride,
               box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// A tensor map only encodes an address and a shape, so one encoded for (X, rows, head_dim)
// serves every later call with the same three: a few recent maps are kept (a decode step
// projects the same small buffers layer after layer).
struct MapCacheEntry {
    const uint16_t* X = nullptr;
    int64_t rows = 0;
    int32_t head_dim = 0;
    CUtensorMap map;
};
constexpr int kMapCache = 64;  // e.g. a decode step: 32 layers, a query and a key buffer each
MapCacheEntry g_map_cache[kMapCache];
int g_map_next = 0;
std::mutex g_map_mu;

bool rows_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const uint16_t* X,
              int64_t rows, int32_t head_dim) {
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        for (const MapCacheEntry& e : g_map_cache) {
            if (e.X == X && e.rows == rows && e.head_dim == head_dim) {
                *map = e.map;
                return true;
            }
        }
    }
    if (!encode_rows_map(enc, map, X, rows, head_dim)) return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    MapCacheEntry& e = g_map_cache[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
    e.X = X;
    e.rows = rows;
    e.head_dim = head_dim;
    e.map = *map;
    return true;
}

}  // namespace

hss_status launch_project2(const ProjectArgs& a0, const ProjectArgs* a1, cudaStream_t stream) {
    const int64_t rows0 = a0.num_rows, rows1 = a1 != nullptr ? a1->num_rows : 0;
    if (rows0 == 0 && rows1 == 0) return HSS_OK;
    const DeviceInfo* dev = current_device_info();
    if (dev == nullptr) return HSS_ERR_CUDA;
    if (!project_shape_supported(a0.head_dim, a0.r)) return HSS_ERR_UNSUPPORTED_SHAPE;
    const ProjLayout L = make_layout(a0.head_dim, a0.r, dev->max_smem_optin);
    if (L.stages < 2) return HSS_ERR_UNSUPPORTED_SHAPE;
    auto enc = encoder();
    if (enc == nullptr) return HSS_ERR_CUDA;

    // Segment 0 is the first non-empty one.
    const ProjectArgs* s0 = rows0 > 0 ? &a0 : a1;
    const ProjectArgs* s1 = rows0 > 0 && rows1 > 0 ? a1 : nullptr;
    CUtensorMap map0, map1;
    if (!rows_map(enc, &map0, s0->X, s0->num_rows, a0.head_dim)) return HSS_ERR_CUDA;
    if (s1 != nullptr) {
        if (!rows_map(enc, &map1, s1->X, s1->num_rows, a0.head_dim)) return HSS_ERR_CUDA;
    } else {
        map1 = map0;
    }
    {
        std::lock_guard<std::mutex> lk(g_smem_mu);
        const int d = dev->device & 63;
        if (g_smem_set[d] < L.total_bytes) {
            if (cudaFuncSetAttribute(project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     L.total_bytes) != cudaSuccess) {
                return HSS_ERR_CUDA;
            }
            g_smem_set[d] = L.total_bytes;
        }
    }
    ProjParams p;
    p.P = a0.P;
    p.head_dim = a0.head_dim;
    p.r = a0.r;
    const ProjectArgs* segs[2] = {s0, s1};
    const ProjectArgs* kv = nullptr;
    for (int i = 0; i < 2; ++i) {
        if (segs[i] == nullptr) {
            p.seg[i] = ProjSegment{0, 0, nullptr, nullptr, nullptr, nullptr, nullptr};
            continue;
        }
        p.seg[i].num_rows = segs[i]->num_rows;
        p.seg[i].tiles = (segs[i]->num_rows + kBM - 1) / kBM;
        p.seg[i].out = segs[i]->out;
        p.seg[i].block_ids = segs[i]->block_ids;
        p.seg[i].slots = segs[i]->slots;
        p.seg[i].cache = segs[i]->cache;
        p.seg[i].X = segs[i]->X;
        if (segs[i]->block_ids != nullptr || segs[i]->slots != nullptr) kv = segs[i];
    }
    p.num_kv_heads = kv != nullptr ? kv->num_kv_heads : 1;
    p.block_size = kv != nullptr ? kv->block_size : 1;
    p.max_blocks = kv != nullptr ? kv->max_blocks : 0;
    p.layer_slots = kv != nullptr ? static_cast<int64_t>(kv->layer) * kv->max_blocks : 0;
    p.dev_status = kv != nullptr ? kv->dev_status : nullptr;
    p.lib_error = dev->error_word;
    const int64_t num_tiles = p.seg[0].tiles + p.seg[1].tiles;
    const int grid = static_cast<int>(std::min<int64_t>(num_tiles, 2 * dev->num_sms));
    // A CTA takes at most ceil(num_tiles / grid) tiles: more stages than that would only hold
    // shared memory.  With one tile (a decode step's new block) two stages need 75 KiB instead
    // of 206, so the CTA fits beside a decode scorer's CTA and can do its set-up while that
    // grid finishes.  At most three stages: two CTAs per SM.
    const int64_t per_cta = (num_tiles + grid - 1) / grid;
    const int stages = static_cast<int>(
        std::max<int64_t>(2, std::min<int64_t>(std::min(L.stages, 3), per_cta)));
    const int smem_bytes = L.total_bytes - (L.stages - stages) * L.stage_bytes;
    if (launch_pdl(project_kernel, dim3(grid), dim3(kThreads), smem_bytes, stream, map0, map1,
                   p, stages) != cudaSuccess)
        return HSS_ERR_CUDA;
    return HSS_OK;
}

hss_status launch_project(const ProjectArgs& a, cudaStream_t stream) {
    return launch_project2(a, nullptr, stream);
}

}  // namespace hss
