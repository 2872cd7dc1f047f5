// Short sequences (at most p.short_len = 8 tokens): the whole scan by the
// "Per-token recurrence" of the Modular page "mamba2_ssd_scan", token by
// token, for every (sequence, head):
//
//   dt_t = softplus(dt + dt_bias);   dA_t = exp(A[h] dt_t)
//   S    = S dA_t + dt_t x_t (x) B_t          S from the initial state (or 0)
//   y_t  = C_t . S + D[h] x_t
//   final state <- S
//
// A short sequence's cost is its state: the pool slot read (with an initial
// state) and written, head_dim x dstate values per head, against a few tokens
// of x, B, C and y.  The chunked kernels would also write and re-read a block
// state and an entering state for it; here the state stays in registers and
// the slot is streamed once with 16-byte accesses (serving batches, where most
// sequences are a few tokens long, are bound by exactly this read-modify-
// write: the decode note of the page "Mamba2SSDChunkScanVarlenFwdInplace").
//
// A persistent grid walks the (short sequence, head) items of the list the
// chunk-state kernel's bookkeeping CTA wrote (so no CTA is spent on a longer
// sequence); the chunked kernels skip the short sequences.  Each thread holds 8
// consecutive dstate values of four head_dim rows; the lanes of a row (2 to 32)
// reduce C_t . S with shuffles.  An item's B, C, x and processed dt
// are staged in shared memory first, every thread's loads issued together.
#include "kernels.cuh"
#include "ssd_device.cuh"
#include "trace.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerThread = 4;
constexpr int kNpt = 8;   // dstate values per lane (dstate is a multiple of 16)

// The state of kRowsPerThread head_dim rows from row0 on (kNpt dstate values
// each, from lane `lr`'s column) into registers; rows past head_dim read as 0.
__device__ __forceinline__ void load_rows(const ScanParams &p, int h, int row0, int tid,
                                          int64_t init, float (&s)[kRowsPerThread][kNpt],
                                          int (&pr)[kRowsPerThread], bool (&ok)[kRowsPerThread])
{
    const int L = p.N / kNpt;
    const int n0 = (tid % L) * kNpt;
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        pr[r] = row0 + (tid / L) * kRowsPerThread + r;
        ok[r] = pr[r] < p.P;
        const int64_t off = (static_cast<int64_t>(h) * p.P + (ok[r] ? pr[r] : 0)) * p.N + n0;
#pragma unroll
        for (int k = 0; k < kNpt; k += 4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ok[r] && init >= 0)
                v = load_init4(p, init + off + k);
            s[r][k] = v.x;
            s[r][k + 1] = v.y;
            s[r][k + 2] = v.z;
            s[r][k + 3] = v.w;
        }
    }
}

// One (short sequence, head): the first rows' state loads are issued, then the
// inputs are staged (both latencies overlap), then the recurrence.
__device__ __forceinline__ void scan_one(const ScanParams &p, const SeqRec &rec, int h, int tid,
                                         float *sB, float *sC, float *sX, float *sDt, float *sDA)
{
    const int t0 = rec.t0, len = rec.len;
    const int g = h / (p.H / p.G);
    const int64_t init = rec.init, fin = rec.fin;
    // kNpt consecutive dstate values per lane, L = N / kNpt lanes per head_dim
    // row (a power of two, 2..32), kRowsPerThread rows per thread: a pass covers
    // kThreads / L * kRowsPerThread rows with all their loads in flight at once
    const int L = p.N / kNpt;
    const int rows_per_pass = kThreads / L * kRowsPerThread;
    const int lr = tid % L;    // lane within the row
    const int n0 = lr * kNpt;
    float s[kRowsPerThread][kNpt];
    int pr[kRowsPerThread];
    bool ok[kRowsPerThread];   // uniform over a row's lanes
    load_rows(p, h, 0, tid, init, s, pr, ok);

    // staging, in rounds of 8 elements per thread whose loads are all issued
    // before any is stored
    constexpr int kRound = 8;
    for (int base = 0; base < len * p.N; base += kRound * kThreads) {
        __nv_bfloat16 vb[kRound], vc[kRound];
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            const int i = base + tid + k * kThreads;
            if (i < len * p.N) {
                const int64_t tok = t0 + i / p.N;
                const int64_t col = static_cast<int64_t>(g) * p.N + i % p.N;
                vb[k] = p.B[tok * p.B_ts + col];
                vc[k] = p.C[tok * p.C_ts + col];
            }
        }
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            const int i = base + tid + k * kThreads;
            if (i < len * p.N) {
                sB[i] = __bfloat162float(vb[k]);
                sC[i] = __bfloat162float(vc[k]);
            }
        }
    }
    {
        __nv_bfloat16 vx[kRound];
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            const int i = tid + k * kThreads;
            if (i < len * p.P)
                vx[k] = p.x[(t0 + i / p.P) * p.x_ts + static_cast<int64_t>(h) * p.P + i % p.P];
        }
        float d = 0.f;
        if (tid < len)
            d = processed_dt(p, t0 + tid, h);
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            const int i = tid + k * kThreads;
            if (i < len * p.P)
                sX[i] = __bfloat162float(vx[k]);
        }
        if (tid < len) {
            sDt[tid] = d;
            sDA[tid] = expf(p.A[h] * d);
        }
    }
    __syncthreads();

    const float Dh = p.D ? p.D[h] : 0.f;
    for (int row0 = 0;;) {
        for (int t = 0; t < len; ++t) {
            const float a = sDA[t];
            float bt[kNpt], ct[kNpt];
#pragma unroll
            for (int k = 0; k < kNpt; k += 4) {
                const float4 vb = *reinterpret_cast<const float4 *>(sB + t * p.N + n0 + k);
                const float4 vc = *reinterpret_cast<const float4 *>(sC + t * p.N + n0 + k);
                bt[k] = vb.x; bt[k + 1] = vb.y; bt[k + 2] = vb.z; bt[k + 3] = vb.w;
                ct[k] = vc.x; ct[k + 1] = vc.y; ct[k + 2] = vc.z; ct[k + 3] = vc.w;
            }
            float part[kRowsPerThread], xv[kRowsPerThread];
#pragma unroll
            for (int r = 0; r < kRowsPerThread; ++r) {
                xv[r] = ok[r] ? sX[t * p.P + pr[r]] : 0.f;
                const float w = sDt[t] * xv[r];
                part[r] = 0.f;
#pragma unroll
                for (int k = 0; k < kNpt; ++k) {
                    s[r][k] = fmaf(s[r][k], a, w * bt[k]);
                    part[r] = fmaf(ct[k], s[r][k], part[r]);
                }
            }
            for (int o = L >> 1; o > 0; o >>= 1)
#pragma unroll
                for (int r = 0; r < kRowsPerThread; ++r)
                    part[r] += __shfl_xor_sync(0xffffffffu, part[r], o);
            if (lr == 0) {
#pragma unroll
                for (int r = 0; r < kRowsPerThread; ++r)
                    if (ok[r])
                        p.y[(t0 + t) * p.y_ts + static_cast<int64_t>(h) * p.P + pr[r]] =
                            __float2bfloat16_rn(part[r] + Dh * xv[r]);
            }
        }
        if (fin >= 0) {
#pragma unroll
            for (int r = 0; r < kRowsPerThread; ++r) {
                const int64_t off = (static_cast<int64_t>(h) * p.P + pr[r]) * p.N + n0;
#pragma unroll
                for (int k = 0; k < kNpt; k += 4)
                    if (ok[r])
                        store_final4(p, fin + off + k,
                                     make_float4(s[r][k], s[r][k + 1], s[r][k + 2], s[r][k + 3]));
            }
        }
        row0 += rows_per_pass;
        if (row0 >= p.P)
            break;
        load_rows(p, h, row0, tid, init, s, pr, ok);
    }
}

__global__ void __launch_bounds__(kThreads, 3) short_scan_kernel(ScanParams p)
{
    __shared__ __align__(16) float sB[kShortLenMax * SSD_MAX_DSTATE];
    __shared__ __align__(16) float sC[kShortLenMax * SSD_MAX_DSTATE];
    __shared__ float sX[kShortLenMax * 128];
    __shared__ float sDt[kShortLenMax], sDA[kShortLenMax];

    // the chunk-state kernel has checked query_start_loc and listed the short
    // sequences; only then is anything read or written
    pdl_wait();
    if (!p.hdr->valid)
        return;
    const int n_items = p.hdr->n_short * p.H;
    const int tid = threadIdx.x;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const SeqRec rec = p.short_list[item / p.H];
        __syncthreads();   // the previous item's staged inputs are no longer read
        scan_one(p, rec, item % p.H, tid, sB, sC, sX, sDt, sDA);
    }
}

}  // namespace

cudaError_t launch_short_scan(const ScanParams &p, cudaStream_t stream, bool programmatic)
{
    cudaLaunchConfig_t cfg = {};
    // a persistent grid over the (short sequence, head) items the chunk-state
    // kernel listed: about three CTAs per SM, fewer for small batches
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t items = static_cast<int64_t>(p.batch) * p.H;
    cfg.gridDim = dim3(static_cast<unsigned>(items < 3 * sms ? items : 3 * sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, short_scan_kernel, p);
}

}  // namespace ssd
