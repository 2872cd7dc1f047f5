// Stages 1 and 2c: per (chunk, head)
//
//   dt_j    = softplus(dt[j,h] + dt_bias[h])       ("Per-token recurrence",
//   a_j     = A[h] * dt_j                            Modular page "mamba2_ssd_scan")
//   Acum_j  = a_0 + ... + a_j                      (inclusive, within the chunk)
//   S_c     = sum_j exp(Acum_last - Acum_j) dt_j  x_j (x) B_j      (chunk state)
//
// The chunk state is the "chunk-state" part of the chunked SSD form named on
// the kernelindex page "Mamba chunk scan with segsum" and on the module page.
// It is a dense contraction over the chunk's tokens and runs on the tcgen05
// tensor cores:  S_c^T[n, p] = sum_j Bmat[j, n] * (w_j x[j, p]),  M = dstate
// (tiles of 128), N = head_dim, K = tokens.  Bmat arrives by TMA (MN-major,
// 128-byte swizzle).  The weighted operand w_j x[j,p] is formed by the CTA's
// threads and split into bf16 hi + lo parts (two MMAs into one fp32
// accumulator), which keeps the chunk state at fp32-level accuracy: a single
// bf16 rounding of w_j x_j leaves ~1e-3 relative error in the final state.
#include "kernels.cuh"
#include "sm100_ptx.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kKB = 64;              // tokens per K block
constexpr int kBlockBytes = kKB * 128; // one 64-wide, 64-row swizzled block (8 KB)

struct K1Layout {
    uint32_t sB, sHi, sLo, sDt, sAcum, sW, bars, tmem_slot, misc, total;
};

__host__ __device__ inline K1Layout k1_layout(int P_pad, int n_mtiles, int Q)
{
    K1Layout L;
    uint32_t off = 0;
    L.sB = off;
    off += n_mtiles * 2 * kBlockBytes;
    L.sHi = off;
    off += (P_pad / 64) * kBlockBytes;
    L.sLo = off;
    off += (P_pad / 64) * kBlockBytes;
    L.sDt = off;
    off += Q * 4;
    L.sAcum = off;
    off += Q * 4;
    L.sW = off;
    off += Q * 4;
    L.bars = (off + 7) & ~7u;
    off = L.bars + 2 * 8;
    L.tmem_slot = off;
    off += 4;
    L.misc = off;
    off += 64;
    L.total = off;
    return L;
}

__device__ __forceinline__ float softplus_f32(float v)
{
    return v > 20.f ? v : log1pf(expf(v));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

__global__ void __launch_bounds__(kThreads)
    chunk_state_kernel(const __grid_constant__ CUtensorMap tmB, ScanParams p, int P_pad,
                       int n_mtiles, uint32_t tmem_cols)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const K1Layout L = k1_layout(P_pad, n_mtiles, p.Q);
    uint8_t *sB = smem + L.sB;
    uint8_t *sHi = smem + L.sHi;
    uint8_t *sLo = smem + L.sLo;
    float *sDt = reinterpret_cast<float *>(smem + L.sDt);
    float *sAcum = reinterpret_cast<float *>(smem + L.sAcum);
    float *sW = reinterpret_cast<float *>(smem + L.sW);
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
    int *s_abort = reinterpret_cast<int *>(smem + L.misc);
    float *s_warp = reinterpret_cast<float *>(smem + L.misc + 4);  // 8 floats

    const int c = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Nothing to do past the table, and once any CTA has given up on a wait the
    // call is already failed: later CTAs leave at once.
    if (!p.hdr->valid || c >= p.hdr->nchunks || (*(volatile uint32_t *)&p.hdr->errors & kErrTimeout))
        return;
    const ChunkEntry ce = p.chunks[c];
    const int t0 = ce.y, len = ce.z;
    const int g = h / (p.H / p.G);
    const int Q = p.Q;

    if (tid == 0) {
        ptx::mbar_init(bar_tma, 1);
        ptx::mbar_init(bar_mma, 1);
        ptx::fence_barrier_init();
        *s_abort = 0;
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 0) {
        ptx::tmem_alloc(tmem_slot, tmem_cols);
        ptx::tmem_relinquish();
    }

    // ---- dt, softplus, inclusive cumsum of A*dt within the chunk ----
    float d = 0.f, a = 0.f;
    if (tid < len) {
        float v = __bfloat162float(p.dt[static_cast<int64_t>(t0 + tid) * p.H + h]);
        if (p.dt_bias)
            v += p.dt_bias[h];
        d = p.dt_softplus ? softplus_f32(v) : v;
        a = p.A[h] * d;
    }
    float incl = a;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += t;
    }
    if (lane == 31)
        s_warp[warp] = incl;
    __syncthreads();
    float before = 0.f;
    for (int w = 0; w < warp; ++w)
        before += s_warp[w];
    const float acum = before + incl;
    if (tid < Q) {
        sDt[tid] = d;
        sAcum[tid] = acum;
        const int64_t o = (static_cast<int64_t>(c) * p.H + h) * Q + tid;
        p.dtp[o] = d;
        p.acum[o] = acum;
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const float a_last = sAcum[len - 1];
    if (tid < Q)
        sW[tid] = tid < len ? expf(a_last - sAcum[tid]) * sDt[tid] : 0.f;
    __syncthreads();

    const uint32_t idesc = ptx::idesc_bf16_f32(128, P_pad, 1, 1);
    const int nkb = (len + kKB - 1) / kKB;
    const int pchunks = P_pad / 8;  // 16-byte chunks per token row
    const int64_t x_row = static_cast<int64_t>(p.H) * p.P;
    bool failed = false;

    for (int kb = 0; kb < nkb; ++kb) {
        if (tid == 0) {
            ptx::mbar_arrive_expect_tx(bar_tma, n_mtiles * 2 * kBlockBytes);
            for (int nb = 0; nb < n_mtiles * 2; ++nb)
                ptx::tma_load_3d(sB + nb * kBlockBytes, &tmB, bar_tma, nb * 64, g, t0 + kb * kKB);
        }
        // weighted input rows kb*64 .. kb*64+63, split into bf16 hi + lo
        for (int item = tid; item < kKB * pchunks; item += kThreads) {
            const int r = item / pchunks, ch = item % pchunks;
            const int j = kb * kKB + r;
            const int p0 = ch * 8;
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                v[k] = 0.f;
            if (j < len && p0 < p.P) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(
                    p.x + static_cast<int64_t>(t0 + j) * x_row + static_cast<int64_t>(h) * p.P + p0);
                const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(&raw);
                const float w = sW[j];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    v[k] = w * __bfloat162float(xb[k]);
            }
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * k]);
                const __nv_bfloat16 h1 = __float2bfloat16_rn(v[2 * k + 1]);
                hi[k] = pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
                lo[k] = pack_bf16(v[2 * k] - __bfloat162float(h0), v[2 * k + 1] - __bfloat162float(h1));
            }
            const uint32_t off = (p0 / 64) * kBlockBytes + (r >> 3) * 1024 + (r & 7) * 128 +
                                 ((((p0 & 63) >> 3) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4 *>(sHi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(sLo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        ptx::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            if (!ptx::mbar_wait(bar_tma, kb & 1, kWaitTimeoutNs)) {
                *s_abort = 1;
            } else {
                ptx::tc_fence_after_sync();
                const uint32_t aB = ptx::smem_u32(sB), aHi = ptx::smem_u32(sHi),
                               aLo = ptx::smem_u32(sLo);
                for (int mt = 0; mt < n_mtiles; ++mt) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t da = ptx::sdesc_sw128(aB + mt * 2 * kBlockBytes + ks * 2048,
                                                             kBlockBytes, 1024);
                        const uint64_t dh = ptx::sdesc_sw128(aHi + ks * 2048, kBlockBytes, 1024);
                        const uint64_t dl = ptx::sdesc_sw128(aLo + ks * 2048, kBlockBytes, 1024);
                        const uint32_t dt_addr = tmem + mt * P_pad;
                        ptx::mma_bf16_ss(dt_addr, da, dh, idesc, (kb | ks) != 0);
                        ptx::mma_bf16_ss(dt_addr, da, dl, idesc, 1);
                    }
                }
                ptx::mma_commit(bar_mma);
                if (!ptx::mbar_wait(bar_mma, kb & 1, kWaitTimeoutNs))
                    *s_abort = 1;
            }
        }
        __syncthreads();
        if (*s_abort) {
            failed = true;
            break;
        }
    }

    if (!failed) {
        ptx::tc_fence_after_sync();
        const int q = warp & 3, half = warp >> 2;
        const int ncols = P_pad / 2;
        for (int mt = 0; mt < n_mtiles; ++mt) {
            const int n = mt * 128 + q * 32 + lane;
            for (int col = half * ncols; col < (half + 1) * ncols; col += 16) {
                float v[16];
                ptx::tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + mt * P_pad + col, v);
                if (n < p.N) {
                    float *dst = p.schunk +
                                 ((static_cast<int64_t>(c) * p.H + h) * p.P) * p.N + n;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int pp = col + k;
                        if (pp < p.P)
                            dst[static_cast<int64_t>(pp) * p.N] = v[k];
                    }
                }
            }
        }
    } else if (tid == 0) {
        record_error(p.hdr, kErrTimeout);
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, tmem_cols);
    }
}

inline int mtiles_of(int N) { return (N + 127) / 128; }

inline uint32_t pow2_cols(uint32_t v)
{
    uint32_t c = 32;
    while (c < v)
        c <<= 1;
    return c;
}

SmemOptIn s_smem_configured;

}  // namespace

size_t chunk_state_smem_bytes(const ScanParams &p)
{
    return k1_layout(pad64(p.P), mtiles_of(p.N), p.Q).total + 1024;
}

cudaError_t launch_chunk_state(const ScanParams &p, const ChunkStateMaps &maps,
                               cudaStream_t stream)
{
    const int P_pad = pad64(p.P);
    const int n_mtiles = mtiles_of(p.N);
    const uint32_t cols = pow2_cols(static_cast<uint32_t>(n_mtiles * P_pad));
    const size_t smem = chunk_state_smem_bytes(p);
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void *>(chunk_state_kernel), s_smem_configured);
    if (e != cudaSuccess)
        return e;
    dim3 grid(p.max_chunks, p.H);
    chunk_state_kernel<<<grid, kThreads, smem, stream>>>(maps.B, p, P_pad, n_mtiles, cols);
    return cudaGetLastError();
}

}  // namespace ssd
