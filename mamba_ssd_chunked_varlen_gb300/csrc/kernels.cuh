// Host-side launchers of the four scan stages (one translation unit each).
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"

namespace ssd {

// Stage 0: chunk table from query_start_loc, device-side argument checks.
cudaError_t launch_chunk_table(const ScanParams &p, cudaStream_t stream);

// Stage 1+2c: per (chunk, head) processed dt, cumulative log-decay and the
// chunk state  S_c[p][n] = sum_j exp(Acum_last - Acum_j) dt_j x[j,p] B[j,n].
struct ChunkStateMaps {
    CUtensorMap B;  // bf16 (N, G, T), box {64, 1, 64}, 128-byte swizzle
};
size_t chunk_state_smem_bytes(const ScanParams &p);
cudaError_t launch_chunk_state(const ScanParams &p, const ChunkStateMaps &maps,
                               cudaStream_t stream);

// Stage 3: inter-chunk state passing; writes the state entering every chunk
// and the final state of every sequence into its pool slot.
cudaError_t launch_state_passing(const ScanParams &p, cudaStream_t stream);

// Stage 2a/2b/4: per (chunk, 128-row tile, head) C.B^T, the masked diagonal
// block, the off-diagonal C.S_prev^T term and the D skip; writes y.
struct ChunkScanMaps {
    CUtensorMap C;      // bf16 (N, G, T), box {64, 1, 64}
    CUtensorMap B;      // bf16 (N, G, T), box {64, 1, 64}
    CUtensorMap X;      // bf16 (P, H, T), box {64, 1, 64}
    CUtensorMap Sprev;  // bf16 (N, P, chunks*H), box {64, 64, 1}
};
size_t chunk_scan_smem_bytes(const ScanParams &p);
cudaError_t launch_chunk_scan(const ScanParams &p, const ChunkScanMaps &maps,
                              cudaStream_t stream);

// The whole scan (argument checks, tensor maps, the four launches) on a
// caller-provided scratch buffer; `events` (5 CUDA events) may be null.
ssd_status_t scan_impl(void *y, const void *x, const void *dt, const float *A, const void *B,
                       const void *C, const float *D, const float *dt_bias, float *ssm_pool,
                       const int32_t *query_start_loc, const uint8_t *has_initial_state,
                       const uint32_t *cache_indices, int64_t total_len, int32_t batch,
                       int32_t nheads, int32_t head_dim, int32_t ngroups, int32_t dstate,
                       int64_t max_slots, int32_t chunk_size, int32_t dt_softplus,
                       void *workspace, size_t workspace_bytes, ssd_stream_t stream,
                       void *const *events);

inline int pad64(int v) { return (v + 63) / 64 * 64; }

// Opt-in shared memory per block on sm_100 / sm_103 (227 KB).
constexpr int kMaxSmemPerBlock = 232448;

// Per-device record of whether a kernel's dynamic shared-memory limit has been
// raised to kMaxSmemPerBlock (done once per device and kernel, not per call).
struct SmemOptIn {
    std::atomic<uint8_t> done[64];
};

inline cudaError_t ensure_max_smem(const void *kernel, SmemOptIn &state)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < 64 && state.done[dev].load(std::memory_order_acquire))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemPerBlock);
    if (e == cudaSuccess && dev >= 0 && dev < 64)
        state.done[dev].store(1, std::memory_order_release);
    return e;
}

}  // namespace ssd
