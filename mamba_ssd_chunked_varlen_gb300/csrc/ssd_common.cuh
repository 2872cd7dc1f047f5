// Shared definitions of the scan kernels: launch parameters, workspace layout
// and the chunk table.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace ssd {

// Device-side error flags (same values as SSD_DEVERR_* in include/ssd_scan.h).
constexpr uint32_t kErrBadQsl = 0x1u;
constexpr uint32_t kErrBadSlot = 0x2u;
constexpr uint32_t kErrTimeout = 0x4u;

// Limit for every on-chip wait (mbarrier) before the kernel gives up.
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s

// Header words at the start of the workspace.
struct WsHeader {
    uint32_t errors;   // SSD_DEVERR_* bits of the current call
    int32_t nchunks;   // blocks of the call
    int32_t valid;     // 1 when query_start_loc passed the device checks
    int32_t n_short;   // entries of the short-sequence work list
    int32_t n_long;    // entries of the long-sequence work list
    int32_t pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header size");

// Byte offsets of the workspace regions; every region is 256-byte aligned.
struct WsLayout {
    int64_t max_chunks;
    size_t header, seq_first, short_list, long_list, table, decay, schunk, sexp, sprev, total;
};

// Batches of more sequences than this map their blocks once, in a kernel of
// their own that writes a block table, instead of in every CTA (a scan of
// query_start_loc per CTA costs a round per 512 sequences); so do calls whose
// block kernels run in several waves (each wave would map again).
constexpr int32_t kMapBatchMax = 512;

// Where a block lies, as the block table records it.
struct alignas(16) BlockEntry {
    int32_t seq, t0, len;
    int32_t flags;   // 1: the sequence's first block, 2: its last
};

// One sequence of a work list, resolved by the per-call bookkeeping CTA so
// that a consumer reaches all of it with one 32-byte read.
struct __align__(16) SeqRec {
    int32_t t0, len;          // its tokens
    int32_t c_begin, c_end;   // its blocks
    int64_t init, fin;        // element index of its initial / final state (-1: none)
};
static_assert(sizeof(SeqRec) == 32, "record size");

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Tokens per block: chunks longer than 128 tokens are processed as 128-token
// blocks (the chunked form is exact at any chunk size).
__host__ __device__ inline int32_t block_tokens(int32_t chunk_size)
{
    return chunk_size < 128 ? chunk_size : 128;
}

// Upper bound on the number of blocks.  Only sequences longer than short_len
// tokens are cut into blocks (the short-sequence kernel takes the others), and
// at most n = min(batch, T / (short_len + 1)) sequences are that long, so
//   sum_b ceil(L_b / Q) < T / Q + n <= ceil(T / Q) + n:
// the bound's last block index never holds a block.  At least 1.
__host__ __device__ inline int64_t max_chunks_bound(int64_t T, int32_t batch, int32_t Q,
                                                    int32_t short_len)
{
    const int64_t by_len = T / (static_cast<int64_t>(short_len) + 1);
    const int64_t n_long = by_len < batch ? by_len : batch;
    const int64_t bound = (T + Q - 1) / Q + n_long;
    return bound > 0 ? bound : 1;
}

// Q here is the block size (block_tokens of the chunk size).
__host__ __device__ inline WsLayout ws_layout(int64_t T, int32_t batch, int32_t H, int32_t P,
                                              int32_t N, int32_t Q, int32_t short_len)
{
    WsLayout L;
    L.max_chunks = max_chunks_bound(T, batch, Q, short_len);
    const size_t mc = static_cast<size_t>(L.max_chunks);
    size_t off = 0;
    L.header = off;
    off = align256(off + sizeof(WsHeader));
    L.seq_first = off;
    off = align256(off + sizeof(int32_t) * (static_cast<size_t>(batch) + 1));
    L.short_list = off;
    off = align256(off + sizeof(SeqRec) * static_cast<size_t>(batch));
    L.long_list = off;
    off = align256(off + sizeof(SeqRec) * static_cast<size_t>(batch));
    L.table = off;
    off = align256(off + sizeof(BlockEntry) * mc);
    L.decay = off;
    off = align256(off + sizeof(float) * mc * H);
    L.schunk = off;
    off = align256(off + sizeof(__half) * mc * H * P * N);
    L.sexp = off;
    off = align256(off + sizeof(int8_t) * mc * H * (P / 16) * N);
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
    const __nv_bfloat16 *B, *C;   // read directly only by the short-sequence kernel
    const float *A;
    const float *D;        // may be null
    const float *dt_bias;  // may be null
    // where each sequence's state starts and ends: either the slot pool
    // (in place: pool, cache_idx, max_slots) or, when pool is null, separate
    // per-sequence arrays (init_states may be null: zero initial states)
    void *pool;                // fp32, or bf16 when pool_bf16
    int32_t pool_bf16;         // 1: the pool stores bf16 (the scan accumulates in fp32)
    const uint32_t *cache_idx;
    const float *init_states;  // (batch, H, P, N) or null
    float *final_states;       // (batch, H, P, N)
    const int32_t *qsl;
    const uint8_t *has_init;  // may be null
    int64_t T;
    // elements between consecutive tokens (H*P, H, G*N, G*N, H*P when contiguous;
    // larger for column slices of a wider buffer, e.g. a fused projection output)
    int64_t x_ts, dt_ts, B_ts, C_ts, y_ts;
    int32_t batch, H, P, G, N;
    int32_t Q;            // tokens per block (block_tokens of the chunk size)
    int64_t max_slots;
    int32_t dt_softplus;
    int32_t finish_single;   // 1: the chunk-state kernel finishes one-block sequences
                             // (their final and entering states; state passing skips them)
    int32_t short_len;    // sequences of at most this many tokens go to the short-sequence
                          // kernel (the chunked kernels skip them); 0: none
    int32_t max_chunks;   // upper bound on the number of blocks
    uint32_t test_stall_ns;   // 0; otherwise the chunk-state kernel (or the fused scan)
                              // also waits on an mbarrier that nothing completes, with this
                              // limit, so that the bounded-wait failure path runs (tests)
    // workspace regions
    WsHeader *hdr;
    int32_t *seq_first;   // (batch + 1): first block of each sequence, then the total
    SeqRec *short_list;   // the short sequences (hdr->n_short of them)
    SeqRec *long_list;    // the other sequences (hdr->n_long): state passing's list, or
                          // the fused walk's for batches above kMapBatchMax
    BlockEntry *table;    // per block, when the block-map kernel runs; else null (each
                          // CTA maps its own block)
    float *decay;         // [block][head] exp(sum of A*dt over the block)
    __half *schunk;       // [block][head][P][N] block states (zero initial state) in fp16,
                          // each scaled by 2^sexp of its group of 16 consecutive p
    int8_t *sexp;         // [block][head][P/16][N] those exponents
    __nv_bfloat16 *sprev; // [block][head][P][N] state entering each block (bf16 operand)
};

// Grid of the two block kernels (chunk state and chunk scan): with the block
// table (many-wave calls) it is (head groups, blocks), so that every block's
// CTAs are dispatched before the empty block indices past the call's last
// block (the host's bound counts a partial block for every sequence that may
// be long) and a block's head groups run side by side; without it, (blocks,
// head groups).  gridDim.y is at most 65535.
__host__ __device__ inline bool blocks_on_y(const ScanParams &p)
{
    return p.table != nullptr && p.max_chunks <= 65535;
}


__device__ __forceinline__ void record_error(WsHeader *hdr, uint32_t flag)
{
    atomicOr(&hdr->errors, flag);
}

}  // namespace ssd
