// pkv_decode_step_static: one decode step whose workspace is a fixed array in the library's own device memory.
//
// Some callers cannot call cudaMalloc at the point where they run a decode step: code that runs inside a
// framework's memory pool with no hook for extra buffers, plug-ins whose host application owns every allocation,
// or a serving loop that must not allocate after start-up. For them this entry point takes the same inputs and
// output as pkv_decode_step and keeps the workspace (task list, partial states, status word) in g_scratch below,
// a file-scope device array that every GPU which loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <mutex>

#include "pkv_internal.h"

namespace {

using namespace pkv;

static_assert(PKV_STATIC_SCRATCH_BYTES % kWsAlign == 0, "the scratch size must keep workspace offsets aligned");

// The workspace of every pkv_decode_step_static call on a device. Zero when the module loads.
static __device__ __align__(256) unsigned char g_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_addr[kMaxDevices];
std::mutex g_setup_mu;

// Device address of g_scratch on the current device. In host code the name g_scratch is only a host-side handle
// of the symbol, so the address is taken once per device with cudaGetSymbolAddress while that device is current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_E_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_E_UNSUPPORTED;
    void* p = g_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        p = g_addr[dev].load(std::memory_order_relaxed);
        if (!p) {
            if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return PKV_E_CUDA;
            g_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_decode_step_static(const pkv_plan_t* plan, const pkv_problem* problem, const void* q,
                                      const void* k_pool, const void* v_pool, const int32_t* block_table,
                                      const int32_t* seq_lens_dev, float scale, void* out, uint32_t* status_dev,
                                      void* stream) {
    if (!plan || !problem) return PKV_E_NULLPTR;
    if (plan->ws_bytes < 0 || plan->ws_bytes > (int64_t)PKV_STATIC_SCRATCH_BYTES) return PKV_E_WS_TOO_SMALL;
    if (status_dev && (reinterpret_cast<uintptr_t>(status_dev) % 4) != 0) return PKV_E_ALIGN;
    void* ws = nullptr;
    int rc = scratch_address(&ws);
    if (rc != PKV_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Same validation and kernels as the caller-owned-workspace path, all validated before anything is enqueued.
    // The fused merge's arrival counters must start at zero: a completed step leaves them at zero, but a step
    // that gave up (a timeout, a truncated task list) may not, and no caller can re-initialise this array, so
    // every call clears them first.
    rc = decode_step(plan, problem, q, nullptr, nullptr, k_pool, v_pool, block_table, seq_lens_dev, scale, ws,
                     PKV_STATIC_SCRATCH_BYTES, out, stream, true);
    if (rc != PKV_OK) return rc;
    // The status word is the only other part of the array a step reads before writing it: hand it over, then
    // clear it so the next call starts from zero.
    uint32_t* status = &static_cast<pkv_ws_header*>(ws)->status;
    if (status_dev &&
        cudaMemcpyAsync(status_dev, status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return PKV_E_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return PKV_E_CUDA;
    return PKV_OK;
}
