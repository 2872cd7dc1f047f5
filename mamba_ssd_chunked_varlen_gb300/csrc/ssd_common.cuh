// Shared definitions of the scan kernels: launch parameters, workspace layout
// and the chunk table.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {

// Device-side error flags (same values as SSD_DEVERR_* in include/ssd_scan.h).
constexpr uint32_t kErrBadQsl = 0x1u;
constexpr uint32_t kErrBadSlot = 0x2u;
constexpr uint32_t kErrTimeout = 0x4u;

// Limit for every on-chip wait (mbarrier) before the kernel gives up.
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s

// Chunk table entry: one chunk of one sequence, aligned to the sequence start.
//   x = sequence index, y = first token, z = length (1..chunk_size),
//   w = flags (bit 0: first chunk of its sequence, bit 1: last chunk).
using ChunkEntry = int4;
constexpr int kChunkFirst = 1;
constexpr int kChunkLast = 2;

// Header words at the start of the workspace.
struct WsHeader {
    uint32_t errors;   // SSD_DEVERR_* bits of the current call
    int32_t nchunks;   // chunks in the table
    int32_t valid;     // 1 when query_start_loc passed the device checks
    int32_t pad[61];
};
static_assert(sizeof(WsHeader) == 256, "header size");

// Byte offsets of the workspace regions; every region is 256-byte aligned.
struct WsLayout {
    int64_t max_chunks;
    size_t header, chunks, seq_first, dtp, acum, schunk, sprev, total;
};

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Upper bound on the number of chunks: sum_b ceil(L_b / Q) <= ceil(T / Q) + batch.
__host__ __device__ inline int64_t max_chunks_bound(int64_t T, int32_t batch, int32_t Q)
{
    return (T + Q - 1) / Q + batch;
}

__host__ __device__ inline WsLayout ws_layout(int64_t T, int32_t batch, int32_t H, int32_t P,
                                              int32_t N, int32_t Q)
{
    WsLayout L;
    L.max_chunks = max_chunks_bound(T, batch, Q);
    const size_t mc = static_cast<size_t>(L.max_chunks);
    size_t off = 0;
    L.header = off;
    off = align256(off + sizeof(WsHeader));
    L.chunks = off;
    off = align256(off + sizeof(ChunkEntry) * (mc + 1));
    L.seq_first = off;
    off = align256(off + sizeof(int32_t) * (static_cast<size_t>(batch) + 1));
    L.dtp = off;
    off = align256(off + sizeof(float) * mc * H * Q);
    L.acum = off;
    off = align256(off + sizeof(float) * mc * H * Q);
    L.schunk = off;
    off = align256(off + sizeof(float) * mc * H * P * N);
    L.sprev = off;
    off = align256(off + sizeof(__nv_bfloat16) * mc * H * P * N);
    L.total = off;
    return L;
}

// Everything a kernel needs, passed by value.
struct ScanParams {
    __nv_bfloat16 *y;
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *dt;
    const float *A;
    const float *D;        // may be null
    const float *dt_bias;  // may be null
    float *pool;
    const int32_t *qsl;
    const uint8_t *has_init;  // may be null
    const uint32_t *cache_idx;
    int64_t T;
    int32_t batch, H, P, G, N, Q;
    int64_t max_slots;
    int32_t dt_softplus;
    int32_t max_chunks;
    // workspace regions
    WsHeader *hdr;
    ChunkEntry *chunks;
    int32_t *seq_first;   // (batch + 1): first chunk of each sequence, then the total
    float *dtp;           // [chunk][head][Q] processed dt (0 past the chunk end)
    float *acum;          // [chunk][head][Q] inclusive cumulative A*dt within the chunk
    float *schunk;        // [chunk][head][P][N] chunk states (zero initial state)
    __nv_bfloat16 *sprev; // [chunk][head][P][N] state entering each chunk (bf16 operand)
};

__device__ __forceinline__ void record_error(WsHeader *hdr, uint32_t flag)
{
    atomicOr(&hdr->errors, flag);
}

}  // namespace ssd
