// pa_decode_noalloc: paged decode attention whose scratch lives in one fixed
// device buffer owned by the library, for callers that cannot allocate device
// memory.
//
// Who needs it: code running inside a host framework that has already reserved
// the device's memory for its own pool (a direct cudaMalloc there fails, or
// breaks the framework's accounting), plugin hosts that hand a plugin nothing
// but its input and output pointers, and serving loops that cannot afford a
// cudaMalloc/cudaFree, which may synchronise the device and stall other work.
//
// The buffer below is a file-scope device array, so every GPU that loads this
// library holds PA_NOALLOC_SCRATCH_BYTES of it until the process exits.  Host
// code may not use the array's name as a device address (on the host it names
// a host-side stand-in); the device address is looked up per device with
// cudaGetSymbolAddress, with that device current, on the first call there.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pa.h"

static __device__ __align__(256) unsigned char pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device (looked up once).
cudaError_t scratch_on_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, pa_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const pa_shape* shape, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* context_lens, float scale, void* out,
                                       uint32_t* err_word, void* stream) {
    // pa_decode rejects (PA_ERR_WORKSPACE, nothing enqueued) a buffer below the
    // shape's minimum scratch, and uses fewer run-time balanced chunks when the
    // buffer is below its preferred size.
    if (pa_decode_workspace_bytes(shape) == 0) return PA_ERR_INVALID_ARG;
    void* scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return PA_ERR_CUDA;
    // pa_decode validates everything else and clears the arrival counters in
    // the scratch on `stream` before its kernel, so stale contents left by an
    // earlier call do no harm.
    return pa_decode(shape, q, k_pool, v_pool, block_tables, context_lens, scale, out, scratch,
                     (size_t)PA_NOALLOC_SCRATCH_BYTES, err_word, stream);
}
