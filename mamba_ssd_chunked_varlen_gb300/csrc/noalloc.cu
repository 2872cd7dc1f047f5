// The scan for callers that cannot allocate device memory (a plugin inside a
// host framework that owns all device memory, a serving loop that forbids
// allocation once running).  Its scratch is a fixed array in this file
// instead of a caller-provided workspace; nothing here allocates.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/ssd_scan.h"
#include "kernels.cuh"

namespace {

// Scratch of every ssd_scan_varlen_fwd_noalloc call on a device.  Each GPU
// that loads the library holds it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is a host-side stand-in, not a device address, so it is
// never passed directly.  The address is looked up on every call (the lookup
// allocates nothing): a cached address would go stale if the device's context
// were reset and the library's device code loaded again at another address.
cudaError_t scratch_for_current_device(void **out)
{
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess)
        return e;
    *out = ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" ssd_status_t ssd_scan_varlen_fwd_noalloc(
    void *y, const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, const float *dt_bias, float *ssm_pool, const int32_t *query_start_loc,
    const uint8_t *has_initial_state, const uint32_t *cache_indices, int64_t total_len,
    int32_t batch, int32_t nheads, int32_t head_dim, int32_t ngroups, int32_t dstate,
    int64_t max_slots, int32_t chunk_size, int32_t dt_softplus, ssd_stream_t stream)
{
    const size_t need = ssd_scan_varlen_workspace_size(total_len, batch, nheads, head_dim,
                                                       ngroups, dstate, chunk_size);
    const ssd::StateIO io{ssm_pool, cache_indices, max_slots, nullptr, nullptr, 0};
    if (!ssm_pool && batch > 0)
        return SSD_ERR_INVALID_ARG;
    if (need == 0)  // invalid or unsupported sizes: let the full check name the reason
        return ssd::scan_impl(y, x, dt, A, B, C, D, dt_bias, io, query_start_loc,
                              has_initial_state, total_len, batch, nheads, head_dim, ngroups,
                              dstate, chunk_size, dt_softplus, nullptr, 0, stream, nullptr);
    if (need > SSD_NOALLOC_SCRATCH_BYTES)
        return SSD_ERR_TOO_LARGE;
    if (batch == 0)
        return SSD_OK;
    void *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess)
        return SSD_ERR_CUDA;
    return ssd::scan_impl(y, x, dt, A, B, C, D, dt_bias, io, query_start_loc, has_initial_state,
                          total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size,
                          dt_softplus, scratch, SSD_NOALLOC_SCRATCH_BYTES, stream, nullptr);
}
