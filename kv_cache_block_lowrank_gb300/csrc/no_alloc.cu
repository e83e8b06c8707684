// no_alloc.cu -- hss_layer_step for callers that cannot allocate device memory.
//
// hss_layer_step needs a small workspace (per-sequence completion counters for the victim
// ranking it fuses into the scorer) that the caller allocates.  Some callers cannot call
// cudaMalloc at that point: an engine whose memory arena already owns the GPU's memory and
// forbids allocations after start-up, a library loaded into a host that gives it no
// allocator, or a caller outside any CUDA-aware framework that only holds raw pointers to
// its own buffers.  For them this file keeps the counters in a fixed array of device memory
// that is part of the library itself, so the call needs nothing beyond its inputs and
// outputs.
//
// The array holds the counters of at most kStaticMaxSeqs sequences and the one-sequence
// ranking's 32.25 KiB (48.25 KiB on each GPU that loads the library, held until the process
// exits).  Every call shares it, so calls that
// overlap on the GPU (on different streams, or on one stream without ordering) race.
#include <mutex>

#include "internal.h"

namespace hss {
namespace {

constexpr int kStaticMaxSeqs = HSS_LAYER_STEP_STATIC_MAX_SEQS;

constexpr int kStaticWords = kStaticMaxSeqs + 64 + 2 * 4096;
static __device__ __align__(256) int32_t g_static_counters[kStaticWords];

// Device address of g_static_counters, looked up once per device with that device current
// (the symbol's name in host code is only a stand-in, not an address a kernel can use).  It
// is kept for the life of the process: cudaDeviceReset unloads the module, so a caller that
// resets a device reloads the library before the next call on it.
constexpr int kMaxDevices = 64;
int32_t* g_counters_addr[kMaxDevices] = {nullptr};
std::mutex g_counters_mu;

hss_status counters_for_current_device(int32_t** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HSS_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_counters_mu);
    if (g_counters_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_counters) != cudaSuccess || p == nullptr)
            return HSS_ERR_CUDA;
        g_counters_addr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_counters_addr[dev];
    return HSS_OK;
}

}  // namespace
}  // namespace hss

using namespace hss;

extern "C" {

int32_t hss_layer_step_static_max_seqs(void) { return kStaticMaxSeqs; }

hss_status hss_layer_step_static(const hss_dims* dims, const uint16_t* P, const uint16_t* K_new,
                                 const int32_t* new_ids, int64_t num_new, const uint16_t* Q,
                                 int32_t rows_per_seq, uint16_t* Qp, uint16_t* A_g, int32_t layer,
                                 const int32_t* block_table, const int32_t* seq_offsets,
                                 int32_t num_seqs, int64_t total_blocks, float* scores, int32_t k,
                                 int32_t* victims, int32_t* dev_status, void* stream) {
    if (num_seqs > kStaticMaxSeqs) return HSS_ERR_WORKSPACE_TOO_SMALL;
    if (num_seqs <= 0) {
        return hss_layer_step(dims, P, K_new, new_ids, num_new, Q, rows_per_seq, Qp, A_g, layer,
                              block_table, seq_offsets, num_seqs, total_blocks, scores, k,
                              victims, nullptr, 0, dev_status, stream);
    }
    if (Qp == nullptr) return HSS_ERR_NULL_POINTER;
    // Every check hss_layer_step makes comes first, so that a call that fails enqueues
    // nothing, not even the clear.  The array is 256-byte aligned and large enough, so its
    // own checks pass for any address of that alignment; the check never dereferences it.
    const size_t bytes = static_cast<size_t>(kStaticWords) * sizeof(int32_t);
    LayerStepPlan plan;
    hss_status st = layer_step_check(dims, P, K_new, new_ids, num_new, Q, rows_per_seq, Qp, A_g,
                                     layer, block_table, seq_offsets, num_seqs, total_blocks,
                                     scores, k, victims, reinterpret_cast<const void*>(256),
                                     bytes, &plan);
    if (st != HSS_OK) return st;
    // The array's address (a host-side lookup; nothing is enqueued).
    int32_t* counters = nullptr;
    st = counters_for_current_device(&counters);
    if (st != HSS_OK) return st;
    // The counters must start at zero.  A completed call leaves them zero, but the array
    // outlives every call (and an earlier call may have stopped early), so clear the part
    // this call uses, in stream order.
    if (cudaMemsetAsync(counters, 0, hss_layer_step_workspace_bytes(num_seqs),
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return HSS_ERR_CUDA;
    return hss_layer_step(dims, P, K_new, new_ids, num_new, Q, rows_per_seq, Qp, A_g, layer,
                          block_table, seq_offsets, num_seqs, total_blocks, scores, k, victims,
                          counters, bytes, dev_status, stream);
}

}  // extern "C"
