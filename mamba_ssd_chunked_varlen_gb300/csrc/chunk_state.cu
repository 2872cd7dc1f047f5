// Stages 1 and 2c: per (block, group of heads)
//
//   dt_j    = softplus(dt[j,h] + dt_bias[h])       ("Per-token recurrence",
//   a_j     = A[h] * dt_j                            Modular page "mamba2_ssd_scan")
//   Acum_j  = a_0 + ... + a_j                      (inclusive, within the block)
//   S_c     = sum_j exp(Acum_last - Acum_j) dt_j  x_j (x) B_j      (block state)
//   decay_c = exp(Acum_last)
//
// A block is at most 128 tokens of one sequence, aligned to the sequence start
// (a chunk of the chunked SSD form of the kernelindex page "Mamba chunk scan
// with segsum"; chunks longer than 128 tokens are processed as 128-token
// blocks, which the chunked form allows at any chunk size).
//
// The block state is a dense contraction over the block's tokens and runs on
// the tcgen05 tensor cores, for several heads of one group at once:
//   S^T[n, (h,p)] = sum_j Bmat[j, n] * (w_j,h x[j, h, p])
// M = dstate (tiles of 128), N = heads x head_dim (<= 256), K = tokens.  B and
// x arrive by TMA (MN-major, 128-byte swizzle).  Both operands are turned into
// fp16 in place, each with a power-of-two scale chosen from its largest
// magnitude (largest value in [2^14, 2^15)), so that fp16's range holds them
// and its 11-bit significand rounds w x with relative error <= 2^-11; B itself
// converts exactly.  One bf16 rounding of w x would leave ~1e-3 relative error
// in final states; this leaves ~3e-4.  The scales are removed exactly in the
// epilogue.  The CTA maps its block to its sequence itself, and CTA (0,0)
// writes the per-sequence first-block table and resets the error word.
//
// Block states are stored [block][head][p][n] like the pool's slots, so the
// state-passing kernel reads and writes both with the same coalesced pattern.
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "sm100_ptx.cuh"
#include "ssd_device.cuh"
#include "trace.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 128;                     // tokens per block (max)
constexpr int kNBlockBytes = kRows * 128;      // one 64-wide block of 128 rows (16 KB)

struct K1Layout {
    uint32_t sB, sW, sDt, sAcum, sWt, scratch, bars, tmem_slot, total;
};

__host__ __device__ inline K1Layout k1_layout(int NP, int n_mtiles, int HB)
{
    K1Layout L;
    uint32_t off = 0;
    L.sB = off;
    off += n_mtiles * 2 * kNBlockBytes;
    L.sW = off;
    off += (NP / 64) * kNBlockBytes;
    L.sDt = off;
    off += HB * kRows * 4;
    L.sAcum = off;
    off += HB * kRows * 4;
    L.sWt = off;
    off += HB * kRows * 4;
    L.scratch = off;
    off += 64 * 4;
    L.bars = (off + 7) & ~7u;
    off = L.bars + 4 * 8;
    L.tmem_slot = off;
    off += 16;
    L.total = off;
    return L;
}

// Largest |value| of a CTA-wide set: every thread passes its partial maximum.
__device__ __forceinline__ float block_max(float v, float *s_red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0)
        s_red[warp] = v;
    __syncthreads();
    float m = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w)
        m = fmaxf(m, s_red[w]);
    __syncthreads();
    return m;
}

// Exponent e such that max * 2^e lies in [2^14, 2^15) (0 for max == 0),
// clamped so that the scale stays a finite fp32 power of two.
__device__ __forceinline__ int fp16_scale_exp(float max_abs)
{
    if (!(max_abs > 0.f))
        return 0;
    int ex;
    frexpf(max_abs, &ex);  // max = f * 2^ex, f in [0.5, 1)
    int e = 15 - ex;
    return e > 100 ? 100 : (e < -100 ? -100 : e);
}

__device__ __forceinline__ uint32_t pack_f16(float a, float b)
{
    __half2 t = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

__global__ void __launch_bounds__(kThreads)
    chunk_state_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmX,
                       ScanParams p, int HB, int NP, int n_mtiles, uint32_t tmem_cols)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const K1Layout L = k1_layout(NP, n_mtiles, HB);
    uint8_t *sB = smem + L.sB;
    uint8_t *sW = smem + L.sW;
    float *sDt = reinterpret_cast<float *>(smem + L.sDt);
    float *sAcum = reinterpret_cast<float *>(smem + L.sAcum);
    float *sWt = reinterpret_cast<float *>(smem + L.sWt);
    int32_t *scratch = reinterpret_cast<int32_t *>(smem + L.scratch);
    uint64_t *bar_b = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *bar_x = bar_b + 1;
    uint64_t *bar_mma = bar_b + 2;   // one per state tile (n_mtiles <= 2)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
    float *s_part = reinterpret_cast<float *>(scratch + 40);  // 8 warp partials
    float *s_red = reinterpret_cast<float *>(scratch + 48);   // 8 warp maxima

    const int blk = blockIdx.x;
    const int h0 = blockIdx.y * HB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool leader = blockIdx.x == 0 && blockIdx.y == 0;
    if (tid == 0)
        SSD_TRACE_EV(0, 0);

    if (leader && tid == 0)
        p.hdr->errors = 0u;
    const BlockInfo bi = map_block<kThreads>(p, blk, scratch, leader ? p.seq_first : nullptr);
    if (leader) {
        for (int b = tid; b < p.batch; b += kThreads)
            if (static_cast<int64_t>(p.cache_idx[b]) >= p.max_slots)
                record_error(p.hdr, kErrBadSlot);
        if (tid == 0) {
            if (!bi.valid)
                record_error(p.hdr, kErrBadQsl);
            p.hdr->valid = bi.valid;
            p.hdr->nchunks = bi.valid ? bi.total : 0;
            __threadfence();
        }
    }
    // the state-passing kernel may start launching; it waits for this grid
    pdl_launch_dependents();
    if (!bi.valid || bi.seq < 0)
        return;
    const int t0 = bi.t0, len = bi.len;
    const int g = h0 / (p.H / p.G);
    if (tid == 0)
        SSD_TRACE_EV(0, 1);

    if (tid == 0) {
        ptx::mbar_init(bar_b, 1);
        ptx::mbar_init(bar_x, 1);
        ptx::mbar_init(bar_mma, 1);
        ptx::mbar_init(bar_mma + 1, 1);
        ptx::fence_barrier_init();
        // x rows of the block for the CTA's heads (MN-major, the layout of the
        // weighted operand, which is formed in place)
        ptx::mbar_arrive_expect_tx(bar_x, (NP / 64) * kNBlockBytes);
        for (int cb = 0; cb < NP / 64; ++cb)
            for (int rb = 0; rb < 2; ++rb)
                ptx::tma_load_3d(sW + cb * kNBlockBytes + rb * 64 * 128, &tmX, bar_x,
                                 h0 * p.P + cb * 64, t0 + rb * 64, 0);
        // B rows of the block: n_mtiles*2 blocks of 64 dstate columns x 2 x 64 rows
        ptx::mbar_arrive_expect_tx(bar_b, n_mtiles * 2 * kNBlockBytes);
        for (int nb = 0; nb < n_mtiles * 2; ++nb)
            for (int rb = 0; rb < 2; ++rb)
                ptx::tma_load_3d(sB + nb * kNBlockBytes + rb * 64 * 128, &tmB, bar_b, nb * 64, g,
                                 t0 + rb * 64);
    }
    if (warp == 0) {
        ptx::tmem_alloc(tmem_slot, tmem_cols);
        ptx::tmem_relinquish();
    }

    // ---- dt, softplus, cumulative A*dt per head: every head's dt loaded at
    //      once (one round trip), then two heads per scan pass ----
    const int half = tid >> 7, j = tid & 127;
    float dv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int hh = 2 * k + half;
        dv[k] = (hh < HB && j < len) ? processed_dt(p, t0 + j, h0 + hh) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (2 * k >= HB)
            break;
        const int hh = 2 * k + half;
        const float a = hh < HB ? p.A[h0 + hh] * dv[k] : 0.f;
        const float incl = warp_inclusive_scan(a);
        if (lane == 31)
            s_part[warp] = incl;
        __syncthreads();
        float before = 0.f;
        for (int w = half * 4; w < warp; ++w)
            before += s_part[w];
        if (hh < HB) {
            sDt[hh * kRows + j] = dv[k];
            sAcum[hh * kRows + j] = before + incl;
        }
        __syncthreads();
    }
    float wmax = 0.f;
    for (int i = tid; i < HB * kRows; i += kThreads) {
        const int hh = i / kRows, jj = i % kRows;
        const float last = sAcum[hh * kRows + len - 1];
        const float w = jj < len ? expf(last - sAcum[i]) * sDt[i] : 0.f;
        sWt[i] = w;
        wmax = fmaxf(wmax, fabsf(w));
        if (jj == 0)
            p.decay[static_cast<int64_t>(blk) * p.H + h0 + hh] = expf(last);
    }
    if (tid == 0)
        SSD_TRACE_EV(0, 2);

    bool failed = !(ptx::mbar_wait(bar_x, 0, kWaitTimeoutNs) && ptx::mbar_wait(bar_b, 0, kWaitTimeoutNs));
    failed = __syncthreads_or(failed);
    if (tid == 0)
        SSD_TRACE_EV(0, 3);

    const int chunks8 = NP / 8;            // 16-byte chunks per token row of x
    const int width = HB * p.P;            // valid columns
    const int nbchunks = n_mtiles * 2 * kNBlockBytes / 16;
    int eB = 0, eW = 0;
    if (!failed) {
        // ---- power-of-two scales from the largest |B| and |w| * |x| ----
        float bmax = 0.f, xmax = 0.f;
        for (int c = tid; c < nbchunks; c += kThreads) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(sB + c * 16);
            const __nv_bfloat16 *v = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                bmax = fmaxf(bmax, fabsf(__bfloat162float(v[k])));
        }
        for (int item = tid; item < kRows * chunks8; item += kThreads) {
            const int r = item / chunks8, c0 = (item % chunks8) * 8;
            if (r >= len || c0 >= width)
                continue;
            const uint32_t off = (c0 >> 6) * kNBlockBytes + (r >> 3) * 1024 + (r & 7) * 128 +
                                 ((((c0 & 63) >> 3) ^ (r & 7)) << 4);
            const uint4 raw = *reinterpret_cast<const uint4 *>(sW + off);
            const __nv_bfloat16 *v = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                xmax = fmaxf(xmax, fabsf(__bfloat162float(v[k])));
        }
        bmax = block_max(bmax, s_red);
        xmax = block_max(xmax, s_red);
        wmax = block_max(wmax, s_red);
        if (tid == 0)
            SSD_TRACE_EV(0, 8);
        eB = fp16_scale_exp(bmax);
        eW = fp16_scale_exp(wmax * xmax);
        const float sBsc = ldexpf(1.f, eB), sWsc = ldexpf(1.f, eW);

        // ---- B -> fp16 in place (exact: bf16 significands fit fp16's) ----
        for (int c = tid; c < nbchunks; c += kThreads) {
            uint4 raw = *reinterpret_cast<const uint4 *>(sB + c * 16);
            const __nv_bfloat16 *v = reinterpret_cast<const __nv_bfloat16 *>(&raw);
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                o[k] = pack_f16(__bfloat162float(v[2 * k]) * sBsc, __bfloat162float(v[2 * k + 1]) * sBsc);
            *reinterpret_cast<uint4 *>(sB + c * 16) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (tid == 0)
            SSD_TRACE_EV(0, 9);
        // ---- weighted input w_j x_j -> fp16 in place (zero past the block end) ----
        for (int item = tid; item < kRows * chunks8; item += kThreads) {
            const int r = item / chunks8, c0 = (item % chunks8) * 8;
            const uint32_t off = (c0 >> 6) * kNBlockBytes + (r >> 3) * 1024 + (r & 7) * 128 +
                                 ((((c0 & 63) >> 3) ^ (r & 7)) << 4);
            uint32_t o[4] = {0u, 0u, 0u, 0u};
            if (r < len && c0 < width) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(sW + off);
                const __nv_bfloat16 *v = reinterpret_cast<const __nv_bfloat16 *>(&raw);
                const float w = sWt[(c0 / p.P) * kRows + r] * sWsc;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    o[k] = pack_f16(w * __bfloat162float(v[2 * k]), w * __bfloat162float(v[2 * k + 1]));
            }
            *reinterpret_cast<uint4 *>(sW + off) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    if (tid == 0)
        SSD_TRACE_EV(0, 10);
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0)
        SSD_TRACE_EV(0, 4);

    if (tid == 0 && !failed) {
        const uint32_t idesc = ptx::idesc_f16_f32(128, NP, 1, 1);
        const uint64_t dB0 = ptx::sdesc_sw128(ptx::smem_u32(sB), kNBlockBytes, 1024);
        const uint64_t dW0 = ptx::sdesc_sw128(ptx::smem_u32(sW), kNBlockBytes, 1024);
        const int nks = (len + 15) / 16;
        for (int mt = 0; mt < n_mtiles; ++mt) {
            const uint64_t dBm = ptx::sdesc_add(dB0, mt * 2 * kNBlockBytes);
            ptx::mma_bf16_ss(tmem + mt * NP, dBm, dW0, idesc, 0);
            for (int ks = 1; ks < nks; ++ks)
                ptx::mma_bf16_ss(tmem + mt * NP, ptx::sdesc_add(dBm, ks * 2048),
                                 ptx::sdesc_add(dW0, ks * 2048), idesc, 1);
            // each state tile is stored as soon as its accumulator is final
            ptx::mma_commit(bar_mma + mt);
        }
    }

    if (!failed) {
        // ---- epilogue: S^T tile [n][(h,p)] -> S_c[blk][h][p][n], scales removed ----
        const float unscale_b = ldexpf(1.f, -eB), unscale_w = ldexpf(1.f, -eW);
        const int q = warp & 3, chalf = warp >> 2;
        const int ncols = NP / 2;
        for (int mt = 0; mt < n_mtiles && !failed; ++mt) {
            if (!ptx::mbar_wait(bar_mma + mt, 0, kWaitTimeoutNs)) {
                failed = true;
                break;
            }
            ptx::tc_fence_after_sync();
            const int n = mt * 128 + q * 32 + lane;
            for (int col = chalf * ncols; col < (chalf + 1) * ncols; col += 64) {
                float v[2][32];
                const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) + mt * NP + col;
                ptx::tmem_ld32_pair(ta, ta + 32, v[0], v[1]);
                if (n < p.N) {
                    const float us = unscale_b * unscale_w;
#pragma unroll
                    for (int c16 = 0; c16 < 4; ++c16) {
                        const int c = col + c16 * 16;
                        if (c >= width)
                            continue;
                        // 16 columns never straddle two heads (head_dim % 16 == 0); a
                        // warp writes 32 consecutive n of one p: 128 contiguous bytes
                        const int hh = c / p.P, p0 = c % p.P;
                        float *dst = p.schunk +
                                     ((static_cast<int64_t>(blk) * p.H + h0 + hh) * p.P + p0) * p.N + n;
                        const float *src = &v[c16 >> 1][(c16 & 1) * 16];
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            dst[static_cast<int64_t>(k) * p.N] = src[k] * us;
                    }
                }
            }
        }
    }
    if (failed && tid == 0)
        record_error(p.hdr, kErrTimeout);

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0)
        SSD_TRACE_EV(0, 7);
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, tmem_cols);
    }
}

SmemOptIn s_smem_configured;

}  // namespace

K1Config chunk_state_config(int H, int G, int P, int N)
{
    K1Config c{};
    const int hpg = H / G;
    c.n_mtiles = (N + 127) / 128;
    // heads per CTA: columns of one MMA (<= 128, so that two CTAs share an SM's
    // tensor memory and shared memory), at most 8 heads
    for (int hb = hpg < 8 ? hpg : 8; hb >= 1; --hb) {
        if (hpg % hb)
            continue;
        const int np = pad64(hb * P);
        if (np > 128 && hb > 1)
            continue;
        c.HB = hb;
        c.NP = np;
        break;
    }
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(c.n_mtiles * c.NP))
        cols <<= 1;
    c.tmem_cols = cols;
    c.smem = k1_layout(c.NP, c.n_mtiles, c.HB).total + 1024;
    return c;
}

cudaError_t launch_chunk_state(const ScanParams &p, const ChunkStateMaps &maps,
                               cudaStream_t stream)
{
    const K1Config c = chunk_state_config(p.H, p.G, p.P, p.N);
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void *>(chunk_state_kernel), s_smem_configured);
    if (e != cudaSuccess)
        return e;
    dim3 grid(p.max_chunks, p.H / c.HB);
    chunk_state_kernel<<<grid, kThreads, c.smem, stream>>>(maps.B, maps.X, p, c.HB, c.NP,
                                                           c.n_mtiles, c.tmem_cols);
    return cudaGetLastError();
}

}  // namespace ssd
