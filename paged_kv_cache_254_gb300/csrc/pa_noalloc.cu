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
// a host-side stand-in); the device address is looked up with
// cudaGetSymbolAddress, with the caller's device current, on every call.  The
// lookup is cheap once the module is loaded, and an address cached across
// calls would go stale after a device reset or a primary-context teardown.
#include <cuda_runtime.h>

#include "../../include/pa.h"

static __device__ __align__(256) unsigned char pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace pa {
size_t decode_min_workspace_bytes(const pa_shape* shape, pa_status* why);
}

extern "C" pa_status pa_decode_noalloc(const pa_shape* shape, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* context_lens, float scale, void* out,
                                       uint32_t* err_word, void* stream) {
    // The shape's smallest scratch must fit the buffer; the check comes first,
    // before any pointer is looked at or anything is enqueued.  (A buffer below
    // the preferred size only means fewer run-time balanced chunks.)
    pa_status why = PA_OK;
    const size_t need = pa::decode_min_workspace_bytes(shape, &why);
    if (need == 0) return why;
    if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, pa_noalloc_scratch) != cudaSuccess) return PA_ERR_CUDA;
    // pa_decode validates everything else and clears the part of the scratch
    // that must start at zero on `stream` before its attention kernel, so
    // stale contents left by an earlier call do no harm.
    return pa_decode(shape, q, k_pool, v_pool, block_tables, context_lens, scale, out, scratch,
                     (size_t)PA_NOALLOC_SCRATCH_BYTES, err_word, stream);
}
