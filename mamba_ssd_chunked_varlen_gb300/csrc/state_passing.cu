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
// items of 2048 elements (8 consecutive n per thread) of one (sequence, head);
// the block states (fp16, 16 bytes a thread), their exponents and decays of
// several blocks are loaded before any of them is used.
// Sequences short enough for the short-sequence kernel are not visited.
// L2/HBM-bandwidth bound.  Launched as a programmatic dependent of the
// chunk-state kernel: it waits for that grid before reading.
#include "kernels.cuh"
#include "ssd_device.cuh"
#include "trace.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;

// kAhead blocks' states, exponents and decays are loaded before any of them
// is used.  Long chains (sequences of many blocks) take 8 ahead at up to 128
// registers, two CTAs per SM; calls of short sequences (a few blocks each, so
// a deep prefetch mostly loads past their ends) take 4 ahead at up to 85
// registers, three CTAs per SM, for more items in flight.  A persistent grid
// walks the (sequence, head, element range) items of the sequences the
// chunk-state kernel listed as not short, so a batch of short sequences costs
// no CTA here.  Both forms compute the same values.
template <int kAhead, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks) state_passing_kernel(ScanParams p, int blocks_per_head)
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
        float S[kVec];
        {
            const float4 a = r.init >= 0 ? load_init4(p, r.init + off) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 b = r.init >= 0 ? load_init4(p, r.init + off + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
            S[0] = a.x; S[1] = a.y; S[2] = a.z; S[3] = a.w;
            S[4] = b.x; S[5] = b.y; S[6] = b.z; S[7] = b.w;
        }

        // element index of block c's state of this head: ((c * H) + h) * PN + e;
        // its exponent group: ((c * H) + h) * (P / 16) * N + (p / 16) * N + n
        const int64_t PN16 = PN / 16;
        const int64_t eg = (e / p.N / 16) * p.N + e % p.N;
        int64_t idx = (static_cast<int64_t>(r.c_begin) * p.H + h) * PN + e;
        int64_t idg = (static_cast<int64_t>(r.c_begin) * p.H + h) * PN16 + eg;
        for (int c = r.c_begin; c < r.c_end; c += kAhead) {
            uint4 v[kAhead];
            uint2 ex[kAhead];
            float d[kAhead];
#pragma unroll
            for (int k = 0; k < kAhead; ++k) {
                if (c + k < r.c_end) {
                    v[k] = __ldg(reinterpret_cast<const uint4 *>(p.schunk + idx + k * p.H * PN));
                    ex[k] = __ldg(reinterpret_cast<const uint2 *>(p.sexp + idg + k * p.H * PN16));
                    d[k] = __ldg(p.decay + static_cast<int64_t>(c + k) * p.H + h);
                }
            }
#pragma unroll
            for (int k = 0; k < kAhead; ++k) {
                if (c + k < r.c_end) {
                    uint4 packed;
                    packed.x = pack_bf16(S[0], S[1]);
                    packed.y = pack_bf16(S[2], S[3]);
                    packed.z = pack_bf16(S[4], S[5]);
                    packed.w = pack_bf16(S[6], S[7]);
                    *reinterpret_cast<uint4 *>(p.sprev + idx + k * p.H * PN) = packed;
                    const uint32_t hv[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                    const uint32_t xv[2] = {ex[k].x, ex[k].y};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hv[j]));
                        const uint32_t xw = xv[j >> 1] >> (16 * (j & 1));
                        S[2 * j] = fmaf(d[k], S[2 * j],
                                        f.x * pow2i(-static_cast<int>(static_cast<int8_t>(xw))));
                        S[2 * j + 1] = fmaf(d[k], S[2 * j + 1],
                                            f.y * pow2i(-static_cast<int>(static_cast<int8_t>(xw >> 8))));
                    }
                }
            }
            idx += kAhead * p.H * PN;
            idg += kAhead * p.H * PN16;
        }
        if (fin >= 0) {
            store_final4(p, fin, make_float4(S[0], S[1], S[2], S[3]));
            store_final4(p, fin + 4, make_float4(S[4], S[5], S[6], S[7]));
        }
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
    // one CTA per item up to two (three) per SM, the register limit, each
    // looping over items beyond that; sequences of at most 4 blocks on
    // average take the shallow form
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool shallow = p.T <= 4 * static_cast<int64_t>(p.Q) * p.batch;
    const int64_t items = static_cast<int64_t>(blocks_per_head) * p.batch * p.H;
    const int64_t cap = (shallow ? 3 : 2) * static_cast<int64_t>(sms);
    cfg.gridDim = dim3(static_cast<unsigned>(items < cap ? items : cap));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (shallow)
        return cudaLaunchKernelEx(&cfg, state_passing_kernel<4, 3>, p, blocks_per_head);
    return cudaLaunchKernelEx(&cfg, state_passing_kernel<8, 2>, p, blocks_per_head);
}

}  // namespace ssd
