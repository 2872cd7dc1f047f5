// Stage 0: split every sequence [qsl[b], qsl[b+1]) into chunks of at most
// chunk_size tokens aligned to the sequence start, so that no chunk crosses a
// query_start_loc boundary (the reset rule of the "Per-token recurrence"
// section, Modular page "mamba2_ssd_scan": no cross-sequence bleed), and
// check the device-resident arguments.  One CTA; no host synchronisation.
#include "kernels.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 1024;

__device__ int block_exclusive_scan(int v, int *warp_sums, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += t;
    }
    if (lane == 31)
        warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o)
                s += t;
        }
        warp_sums[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - v;
    *total = warp_sums[31];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kThreads) chunk_table_kernel(ScanParams p)
{
    __shared__ int s_bad;
    __shared__ int s_warp_sums[32];
    const int tid = threadIdx.x;
    if (tid == 0) {
        p.hdr->errors = 0u;
        s_bad = (p.qsl[0] != 0 || static_cast<int64_t>(p.qsl[p.batch]) != p.T) ? 1 : 0;
    }
    __syncthreads();
    for (int b = tid; b < p.batch; b += kThreads) {
        if (p.qsl[b + 1] < p.qsl[b])
            s_bad = 1;
        if (static_cast<int64_t>(p.cache_idx[b]) >= p.max_slots)
            record_error(p.hdr, kErrBadSlot);
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            record_error(p.hdr, kErrBadQsl);
            p.hdr->valid = 0;
            p.hdr->nchunks = 0;
        }
        return;
    }

    int carry = 0;
    for (int base = 0; base < p.batch; base += kThreads) {
        const int b = base + tid;
        int len = 0, n = 0, start = 0;
        if (b < p.batch) {
            start = p.qsl[b];
            len = p.qsl[b + 1] - start;
            n = (len + p.Q - 1) / p.Q;
        }
        int total;
        const int first = carry + block_exclusive_scan(n, s_warp_sums, &total);
        if (b < p.batch) {
            p.seq_first[b] = first;
            for (int k = 0; k < n; ++k) {
                const int off = k * p.Q;
                const int flags = (k == 0 ? kChunkFirst : 0) | (k == n - 1 ? kChunkLast : 0);
                p.chunks[first + k] = make_int4(b, start + off, min(p.Q, len - off), flags);
            }
        }
        carry += total;
    }
    if (tid == 0) {
        p.seq_first[p.batch] = carry;
        p.hdr->nchunks = carry;
        p.hdr->valid = 1;
    }
}

}  // namespace

cudaError_t launch_chunk_table(const ScanParams &p, cudaStream_t stream)
{
    chunk_table_kernel<<<1, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ssd
