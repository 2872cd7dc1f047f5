// Stage 3: the inter-chunk state recurrence with exponential decay (the
// "inter-chunk state recurrence" of the kernelindex page "Mamba chunk scan
// with segsum").  For every sequence b and head h:
//
//   S   = has_initial_state[b] ? ssm_pool[slot][h] : 0
//   for each block c of b:  S_prev[c] = S;   S = decay_c * S + S_c[c]
//   ssm_pool[slot][h] = S                      (in-place write-back, page
//                                               "Mamba2SSDChunkScanVarlenFwdInplace")
// or, in the form with separate state arrays, S starts from initial_states[b]
// and ends in final_states[b] (the "mamba2_ssd_scan" module description).
//
// Every (p, n) element is an independent chain, so the grid covers the
// head_dim x dstate elements of every (sequence, head) with 4 elements per
// thread; the block states and decays of several blocks are loaded before
// any of them is used.  L2/HBM-bandwidth bound.  Launched as a programmatic
// dependent of the chunk-state kernel: it waits for that grid before reading.
#include "kernels.cuh"
#include "ssd_device.cuh"
#include "trace.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 4;
constexpr int kAhead = 8;  // blocks loaded ahead of use

// at most 64 registers: two of these CTAs fit beside a chunk-state CTA on an
// SM while they wait for it
__global__ void __launch_bounds__(kThreads, 4) state_passing_kernel(ScanParams p, int blocks_per_head)
{
    if (threadIdx.x == 0)
        SSD_TRACE_EV(1, 0);
    pdl_launch_dependents();
    pdl_wait();
    if (threadIdx.x == 0)
        SSD_TRACE_EV(1, 1);
    if (!p.hdr->valid)
        return;
    const int b = blockIdx.x / blocks_per_head;
    const int blk = blockIdx.x % blocks_per_head;
    const int h = blockIdx.y;
    const int64_t PN = static_cast<int64_t>(p.P) * p.N;
    const int64_t e = (static_cast<int64_t>(blk) * kThreads + threadIdx.x) * kVec;
    if (b >= p.batch || e >= PN)
        return;

    const int64_t init = seq_init_index(p, b), fin = seq_final_index(p, b);
    const int64_t off = static_cast<int64_t>(h) * PN + e;

    float4 S = make_float4(0.f, 0.f, 0.f, 0.f);
    if (init >= 0)
        S = load_init4(p, init + off);

    const int c_begin = p.seq_first[b], c_end = p.seq_first[b + 1];
    const int64_t stride = static_cast<int64_t>(p.H) * PN;
    const float *__restrict__ sc = p.schunk + (static_cast<int64_t>(c_begin) * p.H + h) * PN + e;
    __nv_bfloat16 *__restrict__ sp = p.sprev + (static_cast<int64_t>(c_begin) * p.H + h) * PN + e;
    const float *__restrict__ dec = p.decay + static_cast<int64_t>(c_begin) * p.H + h;
    for (int c = c_begin; c < c_end; c += kAhead) {
        float4 v[kAhead];
        float d[kAhead];
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
            if (c + k < c_end) {
                v[k] = __ldg(reinterpret_cast<const float4 *>(sc + k * stride));
                d[k] = __ldg(dec + static_cast<int64_t>(k) * p.H);
            }
        }
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
            if (c + k < c_end) {
                uint2 packed;
                packed.x = pack_bf16(S.x, S.y);
                packed.y = pack_bf16(S.z, S.w);
                *reinterpret_cast<uint2 *>(sp + k * stride) = packed;
                S.x = fmaf(d[k], S.x, v[k].x);
                S.y = fmaf(d[k], S.y, v[k].y);
                S.z = fmaf(d[k], S.z, v[k].z);
                S.w = fmaf(d[k], S.w, v[k].w);
            }
        }
        sc += kAhead * stride;
        sp += kAhead * stride;
        dec += static_cast<int64_t>(kAhead) * p.H;
    }
    if (fin >= 0)
        store_final4(p, fin + off, S);
    if (threadIdx.x == 0)
        SSD_TRACE_EV(1, 2);
}

}  // namespace

cudaError_t launch_state_passing(const ScanParams &p, cudaStream_t stream, bool programmatic)
{
    const int64_t PN = static_cast<int64_t>(p.P) * p.N;
    const int blocks_per_head = static_cast<int>((PN / kVec + kThreads - 1) / kThreads);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks_per_head) * p.batch, p.H);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, state_passing_kernel, p, blocks_per_head);
}

}  // namespace ssd
