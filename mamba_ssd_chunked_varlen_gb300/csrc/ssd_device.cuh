// Device helpers shared by the scan kernels: programmatic dependent launch,
// block scans, mapping of a block index to its sequence, dt processing.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ssd_common.cuh"

namespace ssd {

// ---------------------------------------------------------------- PDL
// Lets the next kernel in the stream start launching (its CTAs run their
// prologue and then block in pdl_wait()).
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Blocks until the previous kernel in the stream has completed and its memory
// writes are visible (a no-op when the launch was not programmatic).
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ float softplus_f32(float v)
{
    return v > 20.f ? v : log1pf(expf(v));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

// ---------------------------------------------------------------- block states
// Block states cross the workspace as fp16, each group of 16 consecutive p
// (one n) scaled by a power of two 2^k that puts the group's largest magnitude
// in [2^14, 2^15): every value of the group down to 2^-28 of that maximum keeps
// fp16's full 11-bit precision (relative rounding <= 2^-11), and no value
// overflows, whatever the magnitude of the states.  k is stored beside them
// as an int8 per group.
__device__ __forceinline__ int state_group_exp(float maxabs)
{
    const int e = static_cast<int>((__float_as_uint(maxabs) >> 23) & 0xffu);
    if (e == 0 || e == 255)
        return 0;
    return min(max(141 - e, -100), 100);
}

// 2^k for |k| <= 126.
__device__ __forceinline__ float pow2i(int k)
{
    return __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
}

// A group of 16 state values rounded as they cross the workspace: fp16 after
// scaling by the group's exponent, then back.
__device__ __forceinline__ void round_state_group(float (&v)[16])
{
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k)
        m = fmaxf(m, fabsf(v[k]));
    const int ke = state_group_exp(m);
    const float sc = pow2i(ke), inv = pow2i(-ke);
#pragma unroll
    for (int k = 0; k < 16; ++k)
        v[k] = __half2float(__float2half_rn(v[k] * sc)) * inv;
}

// Processed step of token t, head h: softplus(dt + dt_bias) (or dt + dt_bias).
__device__ __forceinline__ float processed_dt(const ScanParams &p, int64_t t, int h)
{
    float v = __bfloat162float(p.dt[t * p.dt_ts + h]);
    if (p.dt_bias)
        v += p.dt_bias[h];
    return p.dt_softplus ? softplus_f32(v) : v;
}

// Inclusive scan over the 32 lanes of a warp.
template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += t;
    }
    return v;
}

// ---------------------------------------------------------------- state I/O
// Element index of sequence b's initial state row (-1: zero initial state).
// In place ("Mamba2SSDChunkScanVarlenFwdInplace"): its pool slot when
// has_initial_state[b] is set and the slot index is in range.  Separate arrays
// (the "mamba2_ssd_scan" final_states form): row b of initial_states unless
// has_initial_state is given and false.
__device__ __forceinline__ int64_t seq_init_index(const ScanParams &p, int b)
{
    const int64_t slot_elems = static_cast<int64_t>(p.H) * p.P * p.N;
    const bool flag = p.has_init == nullptr || p.has_init[b] != 0;
    if (p.pool != nullptr) {
        const uint32_t slot = p.cache_idx[b];
        return (p.has_init != nullptr && flag && static_cast<int64_t>(slot) < p.max_slots)
                   ? static_cast<int64_t>(slot) * slot_elems
                   : -1;
    }
    return (p.init_states != nullptr && flag) ? static_cast<int64_t>(b) * slot_elems : -1;
}

// Element index of the row that receives sequence b's final state (-1: none,
// an out-of-range slot).
__device__ __forceinline__ int64_t seq_final_index(const ScanParams &p, int b)
{
    const int64_t slot_elems = static_cast<int64_t>(p.H) * p.P * p.N;
    if (p.pool != nullptr) {
        const uint32_t slot = p.cache_idx[b];
        return static_cast<int64_t>(slot) < p.max_slots ? static_cast<int64_t>(slot) * slot_elems
                                                         : -1;
    }
    return static_cast<int64_t>(b) * slot_elems;
}

// Four consecutive state elements from the initial-state storage (the pool,
// fp32 or bf16, or initial_states), widened to fp32.
__device__ __forceinline__ float4 load_init4(const ScanParams &p, int64_t i)
{
    if (p.pool == nullptr)
        return *reinterpret_cast<const float4 *>(p.init_states + i);
    if (!p.pool_bf16)
        return *reinterpret_cast<const float4 *>(static_cast<const float *>(p.pool) + i);
    const uint2 raw = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p.pool) + i);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
    const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
    return make_float4(a.x, a.y, c.x, c.y);
}

// Four consecutive final-state elements into their storage (bf16 storage
// rounds to nearest even).
__device__ __forceinline__ void store_final4(const ScanParams &p, int64_t i, float4 v)
{
    if (p.pool == nullptr) {
        *reinterpret_cast<float4 *>(p.final_states + i) = v;
    } else if (!p.pool_bf16) {
        *reinterpret_cast<float4 *>(static_cast<float *>(p.pool) + i) = v;
    } else {
        uint2 packed;
        packed.x = pack_bf16(v.x, v.y);
        packed.y = pack_bf16(v.z, v.w);
        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.pool) + i) = packed;
    }
}

// One state element from the initial-state storage, widened to fp32.
__device__ __forceinline__ float load_init1(const ScanParams &p, int64_t i)
{
    if (p.pool == nullptr)
        return p.init_states[i];
    if (!p.pool_bf16)
        return static_cast<const float *>(p.pool)[i];
    return __bfloat162float(static_cast<const __nv_bfloat16 *>(p.pool)[i]);
}

// One final-state element into its storage (bf16 storage rounds to nearest
// even).
__device__ __forceinline__ void store_final1(const ScanParams &p, int64_t i, float v)
{
    if (p.pool == nullptr)
        p.final_states[i] = v;
    else if (!p.pool_bf16)
        static_cast<float *>(p.pool)[i] = v;
    else
        static_cast<__nv_bfloat16 *>(p.pool)[i] = __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------- block map
// Where a block (at most `blk_len` tokens of one sequence, aligned to the
// sequence start) lies: blocks are numbered sequence after sequence.
struct BlockInfo {
    int32_t seq;     // sequence index, or -1 when the block index is past the end
    int32_t t0;      // first token
    int32_t len;     // tokens in the block (1..blk_len)
    int32_t first;   // 1 when this is the sequence's first block
    int32_t last;    // 1 when this is the sequence's last block
    int32_t valid;   // 0 when query_start_loc failed the checks
    int32_t total;   // number of blocks of the whole call
};

// Maps block `blk` by scanning query_start_loc.  Called by every thread of a
// CTA of kThreads threads (kThreads a multiple of 32, <= 1024); uses `scratch`
// (ints 0-36 of shared memory).  When `seq_first` is non-null the CTA also
// writes every sequence's first block index there (and the total at [batch]),
// and, when `table` is non-null, every block's entry.
// One pass over query_start_loc per kThreads sequences: the checks of its
// first and last entries ride along with the loads of the scan.
template <int kThreads>
__device__ BlockInfo map_block(const ScanParams &p, int64_t blk, int32_t *scratch,
                               int32_t *seq_first, BlockEntry *table = nullptr)
{
    constexpr int kWarps = kThreads / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t *s_warp = scratch;        // kWarps partial sums
    int32_t *s_res = scratch + 32;    // 5 result ints, written by the owning thread
    int32_t carry = 0;
    int bad = 0;
    for (int base = 0; base < p.batch; base += kThreads) {
        const int b = base + tid;
        int32_t start = 0, len = 0, n = 0;
        if (b < p.batch) {
            start = p.qsl[b];
            const int32_t end = p.qsl[b + 1];
            len = end - start;
            if (len < 0 || (b == 0 && start != 0) ||
                (b == p.batch - 1 && static_cast<int64_t>(end) != p.T)) {
                bad = 1;
                len = 0;
            }
            // a sequence short enough for the short-sequence kernel holds no block
            n = len <= p.short_len ? 0 : (len + p.Q - 1) / p.Q;
        }
        const int32_t incl = warp_inclusive_scan(n);
        if (lane == 31)
            s_warp[warp] = incl;
        __syncthreads();
        int32_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int32_t v = s_warp[w];
            before += w < warp ? v : 0;
            total += v;
        }
        const int32_t first = carry + before + incl - n;
        if (b < p.batch) {
            if (seq_first)
                seq_first[b] = first;
            // (a query_start_loc that fails the checks may give any count: the
            // entries stay inside the table, which is then not used)
            if (table && first >= 0)
                for (int32_t k = 0; k < n && first + k < p.max_chunks; ++k)
                    table[first + k] = BlockEntry{b, start + k * p.Q, min(p.Q, len - k * p.Q),
                                                  (k == 0 ? 1 : 0) | (k == n - 1 ? 2 : 0)};
            if (blk >= first && blk < first + n) {
                const int32_t k = static_cast<int32_t>(blk - first);
                s_res[0] = b;
                s_res[1] = start + k * p.Q;
                s_res[2] = min(p.Q, len - k * p.Q);
                s_res[3] = k == 0;
                s_res[4] = k == n - 1;
            }
        }
        carry += total;
        __syncthreads();
    }
    if (seq_first && tid == 0)
        seq_first[p.batch] = carry;
    bad = __syncthreads_or(bad);
    BlockInfo bi;
    bi.valid = !bad;
    bi.total = carry;
    const bool mine = !bad && blk < carry;
    bi.seq = mine ? s_res[0] : -1;
    bi.t0 = mine ? s_res[1] : 0;
    bi.len = mine ? s_res[2] : 0;
    bi.first = mine ? s_res[3] : 0;
    bi.last = mine ? s_res[4] : 0;
    return bi;
}

// The per-call bookkeeping, by one CTA of kThreads threads after its block
// map (which wrote seq_first): the bad-slot checks, the two work lists of
// sequence records (short ones for the short-sequence kernel, the others for
// state passing or the fused walk) and the header (valid flag, block count).
// `scratch` is the block map's shared ints; 38 and 39 are used here.
template <int kThreads>
__device__ void call_bookkeeping(const ScanParams &p, const BlockInfo &bi, int32_t *scratch)
{
    const int tid = threadIdx.x;
    if (p.pool != nullptr)
        for (int b = tid; b < p.batch; b += kThreads)
            if (static_cast<int64_t>(p.cache_idx[b]) >= p.max_slots)
                record_error(p.hdr, kErrBadSlot);
    int32_t *s_count = scratch + 38, *l_count = scratch + 39;   // past map_block's ints
    if (tid == 0) {
        *s_count = 0;
        *l_count = 0;
    }
    __syncthreads();   // also orders map_block's seq_first writes before the reads
    if (bi.valid)
        for (int b = tid; b < p.batch; b += kThreads) {
            SeqRec r;
            r.t0 = p.qsl[b];
            r.len = p.qsl[b + 1] - r.t0;
            r.c_begin = p.seq_first[b];
            r.c_end = p.seq_first[b + 1];
            r.init = seq_init_index(p, b);
            r.fin = seq_final_index(p, b);
            // a sequence of one block may be finished by the chunk-state kernel
            if (r.len <= p.short_len)
                p.short_list[atomicAdd(s_count, 1)] = r;
            else if (!p.finish_single || r.c_end - r.c_begin > 1)
                p.long_list[atomicAdd(l_count, 1)] = r;
        }
    __syncthreads();
    if (tid == 0) {
        p.hdr->n_short = *s_count;
        p.hdr->n_long = *l_count;
        if (!bi.valid)
            record_error(p.hdr, kErrBadQsl);
        p.hdr->valid = bi.valid;
        p.hdr->nchunks = bi.valid ? bi.total : 0;
        __threadfence();
    }
}

// Block `blk` from the block table (the block-map kernel's output; read only
// after that kernel has completed).
__device__ __forceinline__ BlockInfo lookup_block(const ScanParams &p, int64_t blk)
{
    BlockInfo bi;
    bi.valid = p.hdr->valid;
    bi.total = p.hdr->nchunks;
    const bool mine = bi.valid && blk < bi.total;
    const BlockEntry e = mine ? p.table[blk] : BlockEntry{-1, 0, 0, 0};
    bi.seq = e.seq;
    bi.t0 = e.t0;
    bi.len = e.len;
    bi.first = e.flags & 1;
    bi.last = (e.flags >> 1) & 1;
    return bi;
}

}  // namespace ssd
