// Stage 3: the inter-chunk state recurrence with exponential decay (the
// "inter-chunk state recurrence" of the kernelindex page "Mamba chunk scan
// with segsum").  For every sequence b and head h:
//
//   S   = has_initial_state[b] ? ssm_pool[slot][h] : 0
//   for each chunk c of b:  S_prev[c] = S;   S = exp(Acum_last(c)) * S + S_c[c]
//   ssm_pool[slot][h] = S                      (in-place write-back, page
//                                               "Mamba2SSDChunkScanVarlenFwdInplace")
//
// Every (p, n) element is an independent chain, so the grid covers the
// head_dim x dstate elements of every (sequence, head) with 4 elements per
// thread; the per-chunk loads do not depend on the running state and are
// issued ahead of the FMAs.  HBM/L2-bandwidth bound.
#include "kernels.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 4;

__global__ void __launch_bounds__(kThreads) state_passing_kernel(ScanParams p, int blocks_per_head)
{
    if (!p.hdr->valid)
        return;
    const int b = blockIdx.x / blocks_per_head;
    const int blk = blockIdx.x % blocks_per_head;
    const int h = blockIdx.y;
    const int64_t PN = static_cast<int64_t>(p.P) * p.N;
    const int64_t e = (static_cast<int64_t>(blk) * kThreads + threadIdx.x) * kVec;
    if (b >= p.batch || e >= PN)
        return;

    const uint32_t slot = p.cache_idx[b];
    const bool slot_ok = static_cast<int64_t>(slot) < p.max_slots;
    const bool init = slot_ok && p.has_init != nullptr && p.has_init[b] != 0;
    float *pool_h = p.pool + (static_cast<int64_t>(slot) * p.H + h) * PN + e;

    float4 S = make_float4(0.f, 0.f, 0.f, 0.f);
    if (init)
        S = *reinterpret_cast<const float4 *>(pool_h);

    const int c_begin = p.seq_first[b], c_end = p.seq_first[b + 1];
    for (int c = c_begin; c < c_end; ++c) {
        const int64_t off = (static_cast<int64_t>(c) * p.H + h) * PN + e;
        const float4 sc = *reinterpret_cast<const float4 *>(p.schunk + off);
        const int len = p.chunks[c].z;
        const float decay = expf(p.acum[(static_cast<int64_t>(c) * p.H + h) * p.Q + len - 1]);
        __nv_bfloat162 lo = __floats2bfloat162_rn(S.x, S.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(S.z, S.w);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t *>(&lo);
        packed.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(p.sprev + off) = packed;
        S.x = fmaf(decay, S.x, sc.x);
        S.y = fmaf(decay, S.y, sc.y);
        S.z = fmaf(decay, S.z, sc.z);
        S.w = fmaf(decay, S.w, sc.w);
    }
    if (slot_ok)
        *reinterpret_cast<float4 *>(pool_h) = S;
}

}  // namespace

cudaError_t launch_state_passing(const ScanParams &p, cudaStream_t stream)
{
    const int64_t PN = static_cast<int64_t>(p.P) * p.N;
    const int blocks_per_head = static_cast<int>((PN / kVec + kThreads - 1) / kThreads);
    dim3 grid(static_cast<unsigned>(blocks_per_head) * p.batch, p.H);
    state_passing_kernel<<<grid, kThreads, 0, stream>>>(p, blocks_per_head);
    return cudaGetLastError();
}

}  // namespace ssd
