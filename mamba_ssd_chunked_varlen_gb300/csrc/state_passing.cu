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
// Every (p, n) element is an independent chain, so the work is split into
// items of 1024 elements (4 per thread) of one (sequence, head); the block
// states and decays of several blocks are loaded before any of them is used.
// Sequences short enough for the short-sequence kernel are not visited.
// L2/HBM-bandwidth bound.  Launched as a programmatic dependent of the
// chunk-state kernel: it waits for that grid before reading.
#include "kernels.cuh"
#include "ssd_device.cuh"
#include "trace.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 4;
constexpr int kAhead = 8;  // blocks loaded ahead of use

// at most 64 registers: two of these CTAs fit beside a chunk-state CTA on an
// SM while they wait for it.  A persistent grid walks the (sequence, head,
// element range) items of the sequences the chunk-state kernel listed as not
// short, so a batch of short sequences costs no CTA here.
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
    const int64_t PN = static_cast<int64_t>(p.P) * p.N;
    // items fit 32 bits: batch x nheads x (head_dim x dstate / 1024)
    const int per_seq = p.H * blocks_per_head;
    const int n_items = p.hdr->n_long * per_seq;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const SeqRec r = p.long_list[item / per_seq];
        const int h = (item % per_seq) / blocks_per_head;
        const int64_t e = (static_cast<int64_t>(item % blocks_per_head) * kThreads + threadIdx.x) * kVec;
        if (e >= PN)
            continue;
        const int64_t off = static_cast<int64_t>(h) * PN + e;
        const int64_t fin = r.fin >= 0 ? r.fin + off : -1;
        float4 S = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r.init >= 0)
            S = load_init4(p, r.init + off);

        // element index of block c's state of this head: ((c * H) + h) * PN + e
        int64_t idx = (static_cast<int64_t>(r.c_begin) * p.H + h) * PN + e;
        for (int c = r.c_begin; c < r.c_end; c += kAhead) {
            float4 v[kAhead];
            float d[kAhead];
#pragma unroll
            for (int k = 0; k < kAhead; ++k) {
                if (c + k < r.c_end) {
                    v[k] = __ldg(reinterpret_cast<const float4 *>(p.schunk + idx + k * p.H * PN));
                    d[k] = __ldg(p.decay + static_cast<int64_t>(c + k) * p.H + h);
                }
            }
#pragma unroll
            for (int k = 0; k < kAhead; ++k) {
                if (c + k < r.c_end) {
                    uint2 packed;
                    packed.x = pack_bf16(S.x, S.y);
                    packed.y = pack_bf16(S.z, S.w);
                    *reinterpret_cast<uint2 *>(p.sprev + idx + k * p.H * PN) = packed;
                    S.x = fmaf(d[k], S.x, v[k].x);
                    S.y = fmaf(d[k], S.y, v[k].y);
                    S.z = fmaf(d[k], S.z, v[k].z);
                    S.w = fmaf(d[k], S.w, v[k].w);
                }
            }
            idx += kAhead * p.H * PN;
        }
        if (fin >= 0)
            store_final4(p, fin, S);
    }
    if (threadIdx.x == 0)
        SSD_TRACE_EV(1, 2);
}

}  // namespace

cudaError_t launch_state_passing(const ScanParams &p, cudaStream_t stream, bool programmatic)
{
    const int64_t PN = static_cast<int64_t>(p.P) * p.N;
    const int blocks_per_head = static_cast<int>((PN / kVec + kThreads - 1) / kThreads);
    cudaLaunchConfig_t cfg = {};
    // one CTA per item up to four per SM (the register limit), each looping
    // over items beyond that
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t items = static_cast<int64_t>(blocks_per_head) * p.batch * p.H;
    const int64_t cap = 4 * static_cast<int64_t>(sms);
    cfg.gridDim = dim3(static_cast<unsigned>(items < cap ? items : cap));
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
