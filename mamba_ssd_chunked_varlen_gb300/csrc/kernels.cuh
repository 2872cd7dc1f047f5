// Host-side launchers of the four scan stages (one translation unit each).
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"

namespace ssd {

// Stages 1+2c: per (block, head group) processed dt, cumulative log-decay and
// the block state  S_c[p][n] = sum_j exp(Acum_last - Acum_j) dt_j x[j,p] B[j,n];
// also the per-sequence first-block table and the error word.
struct ChunkStateMaps {
    CUtensorMap B;  // bf16 (N, G, T), box {64, 1, 64}, 128-byte swizzle
    CUtensorMap X;  // bf16 (H*P, T, 1), box {64, 64, 1}
};
struct K1Config {
    int HB, NP, n_mtiles;
    uint32_t tmem_cols;
    size_t smem;
};
K1Config chunk_state_config(int H, int G, int P, int N);
cudaError_t launch_chunk_state(const ScanParams &p, const ChunkStateMaps &maps,
                               cudaStream_t stream, bool programmatic);

// Stages 1, 2c and 3 fused (calls of long sequences with many heads): a
// persistent walk over (sequence, head group, dstate tile) items that keeps
// the block states on chip and writes the state entering every block (bf16)
// and every sequence's final state.  Replaces chunk_state + state_passing for
// the calls use_state_walk picks; with at most kMapBatchMax sequences its CTA
// 0 also does the per-call bookkeeping.
struct StateWalkMaps {
    CUtensorMap B;   // bf16 (N, G, T), box {64, 1, 64}, 128-byte swizzle
    CUtensorMap X;   // bf16 (H*P, T, 1), box {64, 64, 1}
    CUtensorMap Dt;  // bf16 (H, T, 1), box {16, 64, 1}, no swizzle (when dt_tma)
    int dt_tma;      // 1: dt rows are 16-byte aligned and go by TMA; 0: plain loads
};
struct WalkConfig {
    int HB;       // heads per item (HB * head_dim <= 128, one B group)
    int NP;       // HB * head_dim padded to 64 (64 or 128 columns)
    int nT;       // 128-row dstate tiles
    size_t smem;
};
WalkConfig state_walk_config(int H, int G, int P, int N, int batch, int sms);
cudaError_t launch_state_walk(const ScanParams &p, const StateWalkMaps &maps, cudaStream_t stream,
                              bool programmatic);
// Whether a call takes the fused walk: every SM gets an item, the sequences
// average at least 2048 tokens, and the block states the split design would
// write and read back exceed the L2.  Uses the current device's SM count and
// L2 size (152 SMs and 126 MB when no device answers).
bool use_state_walk(int64_t T, int32_t batch, int H, int G, int P, int N, int Qb);

// Whether a call maps its blocks once in the block-map kernel: batches of more
// than kMapBatchMax sequences, and calls whose chunk-scan grid would run more
// than four waves of one CTA per SM (a per-CTA block map costs each wave a
// query_start_loc round trip, the block-map kernel one launch).  Uses the current device's SM count (152 when
// no device answers).
bool use_block_table(int64_t T, int32_t batch, int H, int G, int P, int N, int Qb, int short_len);

// Batches of more than kMapBatchMax sequences: one CTA scans query_start_loc
// once, writes the block table and does the per-call bookkeeping; launched
// before the chunk-state kernel (or the fused walk), which then runs as its
// programmatic dependent.
cudaError_t launch_block_map(const ScanParams &p, cudaStream_t stream);

// Stage 3: inter-block state passing; writes the state entering every block
// and the final state of every sequence into its pool slot.  `programmatic`:
// launched as a programmatic dependent of the previous kernel.
cudaError_t launch_state_passing(const ScanParams &p, cudaStream_t stream, bool programmatic);

// Short sequences (<= p.short_len <= kShortLenMax tokens, including empty
// ones): the per-token recurrence on state tiles streamed through shared
// memory, y and the final state written directly.  Launched after the
// bookkeeping's checks.  Its cost grows with the tokens while the
// chunked kernels spend a whole 128-row block on any sequence.  Measured on
// GB300 with batches of 256 sequences of L tokens, 64 heads of 64 x 128, each
// with an initial state: per-token path 598 us at L = 12, 692 us at 13; the
// chunked path 669-672 us for L = 13..20.  The crossover lies between 12 and
// 13.
constexpr int kShortLenMax = 12;
struct ShortScanMaps {
    CUtensorMap X;  // bf16 (H*P, T, 1), box {tile rows, 8, 1}, no swizzle
    CUtensorMap B;  // bf16 (N, G, T), box {N, 1, 8}
    CUtensorMap C;  // bf16 (N, G, T), box {N, 1, 8}
};
int short_scan_tile_rows(int P, int N);
cudaError_t launch_short_scan(const ScanParams &p, const ShortScanMaps &maps, cudaStream_t stream,
                              bool programmatic);

// Stages 2a/2b/4: per (block, head group) C.B^T, the masked diagonal block,
// the off-diagonal C.S_prev^T term and the D skip; writes y.
struct ChunkScanMaps {
    CUtensorMap C;      // bf16 (N, G, T), box {64, 1, 64}
    CUtensorMap B;      // bf16 (N, G, T), box {64, 1, 64}
    CUtensorMap X;      // bf16 (H*P, T, 1), box {64, 64, 1}
    CUtensorMap Sprev;  // bf16 (N, P, blocks*H), box {64, 64, 1}
};
struct K3Config {
    int HB;          // heads per CTA (one group)
    int P_pad, N_pad;
    int n_xb;        // 64-column X blocks a CTA loads (its heads, from a 64-aligned start)
    int YG;          // heads per off-diagonal MMA (their S_prev tiles stacked along N)
    size_t smem;
};
K3Config chunk_scan_config(int H, int G, int P, int N);
cudaError_t launch_chunk_scan(const ScanParams &p, const ChunkScanMaps &maps, cudaStream_t stream,
                              bool programmatic);

// Where the sequences' states start and end: the slot pool (in place, as
// "Mamba2SSDChunkScanVarlenFwdInplace") when pool is set, else separate
// per-sequence arrays (the final_states form of "mamba2_ssd_scan").
struct StateIO {
    void *pool;                   // (max_slots, H, P, N) fp32 (bf16 when pool_bf16) or null
    const uint32_t *cache_indices;
    int64_t max_slots;
    const float *initial_states;  // (batch, H, P, N) or null (zero initial states)
    float *final_states;          // (batch, H, P, N)
    int pool_bf16;                // 1: the pool stores bf16
};

// Elements between consecutive tokens of x, dt, B, C and y (all rows of a
// token stay contiguous); zero entries mean "contiguous".
struct TokenStrides {
    int64_t x, dt, B, C, y;
};

// The whole scan (argument checks, tensor maps, the three launches) on a
// caller-provided scratch buffer; `events` (5 CUDA events) may be null.  With
// `launch` false it stops after every host-side check and tensor-map encoding
// and launches nothing (the status is the one the call would return before
// its first launch).
ssd_status_t scan_impl(void *y, const void *x, const void *dt, const float *A, const void *B,
                       const void *C, const float *D, const float *dt_bias, const StateIO &io,
                       const int32_t *query_start_loc, const uint8_t *has_initial_state,
                       int64_t total_len, int32_t batch, int32_t nheads, int32_t head_dim,
                       int32_t ngroups, int32_t dstate, int32_t chunk_size, int32_t dt_softplus,
                       void *workspace, size_t workspace_bytes, ssd_stream_t stream,
                       void *const *events, const TokenStrides *strides = nullptr,
                       bool launch = true);

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
