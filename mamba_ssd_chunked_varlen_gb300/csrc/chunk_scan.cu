// Stages 2a, 2b and 4: per (chunk, 128-row tile of the chunk, head)
//
//   CB[i,j]   = C_i . B_j                                       (tensor cores)
//   Ldt[i,j]  = CB[i,j] exp(Acum_i - Acum_j) dt_j   for j <= i, else 0
//   Ydiag     = Ldt X                                           (tensor cores)
//   Yoff      = C S_prev^T                                      (tensor cores)
//   y_i       = Ydiag_i + exp(Acum_i) Yoff_i + D[h] x_i         (bf16 out)
//
// These are the intra-chunk "attention-like" diagonal block built from
// segment sums, and the off-diagonal contribution of the state entering the
// chunk, of the kernelindex page "Mamba chunk scan with segsum"; the D skip is
// the last term of the "Per-token recurrence" of the Modular page
// "mamba2_ssd_scan".  C, B, X and S_prev arrive by TMA with 128-byte swizzle;
// the masked, scaled Ldt tile is formed from the CB accumulator (tensor memory)
// by the CTA's threads and stored back to shared memory as a bf16 operand.
// exp(Acum_i - Acum_j) is always formed from a difference of cumulative sums
// (never a ratio of exponentials), so it cannot overflow for A <= 0.
#include "kernels.cuh"
#include "sm100_ptx.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kRowBlock = 64 * 128;  // 64 rows x 128 B swizzled block (8 KB)

struct K3Layout {
    uint32_t sC, sX, sU, sBm, sS, sL, sDt, sAcum, bars, tmem_slot, misc, total;
};

// sC   : 128 rows (i) x N_pad, K-major, N_pad/64 blocks of 16 KB
// sX   : up to 256 rows (j) x P_pad, MN-major, P_pad/64 blocks of jn*128 B
// sU   : union of {sBm: up to 256 rows (j) x 64 (one K block of B), sS: P_pad rows x N_pad}
//        and {sL: 128 rows (i) x up to 256 (j), K-major}
__host__ __device__ inline K3Layout k3_layout(int P_pad, int N_pad, int Q)
{
    K3Layout L;
    uint32_t off = 0;
    L.sC = off;
    off += (N_pad / 64) * 2 * kRowBlock;
    L.sX = off;
    off += (P_pad / 64) * 4 * kRowBlock;
    L.sU = off;
    L.sBm = off;
    L.sS = off + 4 * kRowBlock;
    const uint32_t phase1 = 4 * kRowBlock + (N_pad / 64) * P_pad * 128;
    L.sL = off;
    const uint32_t phase2 = 4 * 2 * kRowBlock;
    off += phase1 > phase2 ? phase1 : phase2;
    L.sDt = off;
    off += Q * 4;
    L.sAcum = off;
    off += Q * 4;
    L.bars = (off + 7) & ~7u;
    off = L.bars + 5 * 8;
    L.tmem_slot = off;
    off += 4;
    L.misc = off;
    off += 16;
    L.total = off;
    return L;
}

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColOff = 256;  // Yoff at 256, Ydiag at 256 + P_pad

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

__global__ void __launch_bounds__(kThreads)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmS, ScanParams p, int P_pad, int N_pad,
                      int n_itiles)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const K3Layout L = k3_layout(P_pad, N_pad, p.Q);
    uint8_t *sC = smem + L.sC;
    uint8_t *sX = smem + L.sX;
    uint8_t *sBm = smem + L.sBm;
    uint8_t *sS = smem + L.sS;
    uint8_t *sL = smem + L.sL;
    float *sDt = reinterpret_cast<float *>(smem + L.sDt);
    float *sAcum = reinterpret_cast<float *>(smem + L.sAcum);
    uint64_t *bar_c = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *bar_x = bar_c + 1;
    uint64_t *bar_s = bar_c + 2;
    uint64_t *bar_b = bar_c + 3;
    uint64_t *bar_m = bar_c + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
    int *s_abort = reinterpret_cast<int *>(smem + L.misc);

    const int c = blockIdx.x / n_itiles, mt = blockIdx.x % n_itiles, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Nothing to do past the table, and once any CTA has given up on a wait the
    // call is already failed: later CTAs leave at once.
    if (!p.hdr->valid || c >= p.hdr->nchunks || (*(volatile uint32_t *)&p.hdr->errors & kErrTimeout))
        return;
    const ChunkEntry ce = p.chunks[c];
    const int t0 = ce.y, len = ce.z;
    const int i0 = mt * 128;
    if (i0 >= len)
        return;
    const int g = h / (p.H / p.G);
    const int Q = p.Q;
    const int jmax = min(len, i0 + 128);
    const int jn = (jmax + 63) / 64 * 64;  // CB columns / diagonal K extent
    const int nkb = N_pad / 64;
    const int npb = P_pad / 64;

    if (tid == 0) {
        for (int k = 0; k < 5; ++k)
            ptx::mbar_init(bar_c + k, 1);
        ptx::fence_barrier_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (tid < Q) {
        const int64_t o = (static_cast<int64_t>(c) * p.H + h) * Q + tid;
        sDt[tid] = p.dtp[o];
        sAcum[tid] = p.acum[o];
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // ---------------- phase 1: CB = C B^T and Yoff = C S_prev^T (one thread) ----
    if (tid == 0) {
        bool ok = true;
        ptx::mbar_arrive_expect_tx(bar_c, nkb * 2 * kRowBlock);
        for (int kb = 0; kb < nkb; ++kb)
            for (int r = 0; r < 2; ++r)
                ptx::tma_load_3d(sC + (kb * 2 + r) * kRowBlock, &tmC, bar_c, kb * 64, g,
                                 t0 + i0 + r * 64);
        ptx::mbar_arrive_expect_tx(bar_x, npb * jn * 128);
        for (int pb = 0; pb < npb; ++pb)
            for (int rb = 0; rb < jn / 64; ++rb)
                ptx::tma_load_3d(sX + pb * jn * 128 + rb * kRowBlock, &tmX, bar_x, pb * 64, h,
                                 t0 + rb * 64);
        ptx::mbar_arrive_expect_tx(bar_s, nkb * P_pad * 128);
        for (int kb = 0; kb < nkb; ++kb)
            for (int pb = 0; pb < npb; ++pb)
                ptx::tma_load_3d(sS + kb * P_pad * 128 + pb * kRowBlock, &tmS, bar_s, kb * 64,
                                 pb * 64, c * p.H + h);

        const uint32_t id_cb = ptx::idesc_bf16_f32(128, jn, 0, 0);
        const uint32_t id_off = ptx::idesc_bf16_f32(128, P_pad, 0, 0);
        const uint32_t aC = ptx::smem_u32(sC), aB = ptx::smem_u32(sBm), aS = ptx::smem_u32(sS);
        for (int kb = 0; kb < nkb && ok; ++kb) {
            ptx::mbar_arrive_expect_tx(bar_b, jn * 128);
            for (int rb = 0; rb < jn / 64; ++rb)
                ptx::tma_load_3d(sBm + rb * kRowBlock, &tmB, bar_b, kb * 64, g, t0 + rb * 64);
            ok = ptx::mbar_wait(bar_b, kb & 1, kWaitTimeoutNs);
            if (ok && kb == 0)
                ok = ptx::mbar_wait(bar_c, 0, kWaitTimeoutNs) &&
                     ptx::mbar_wait(bar_s, 0, kWaitTimeoutNs);
            if (!ok)
                break;
            ptx::tc_fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t da = ptx::sdesc_sw128(aC + kb * 2 * kRowBlock + ks * 32, 16, 1024);
                const uint64_t db = ptx::sdesc_sw128(aB + ks * 32, 16, 1024);
                const uint64_t ds = ptx::sdesc_sw128(aS + kb * P_pad * 128 + ks * 32, 16, 1024);
                ptx::mma_bf16_ss(tmem, da, db, id_cb, (kb | ks) != 0);
                ptx::mma_bf16_ss(tmem + kColOff, da, ds, id_off, (kb | ks) != 0);
            }
            ptx::mma_commit(bar_m);
            ok = ptx::mbar_wait(bar_m, kb & 1, kWaitTimeoutNs);
        }
        if (!ok)
            *s_abort = 1;
    }
    __syncthreads();

    const int q = warp & 3, half = warp >> 2;
    const int i_loc = q * 32 + lane;
    const int i = i0 + i_loc;  // chunk-local row
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const float ai = sAcum[min(i, Q - 1)];

    if (!*s_abort) {
        // ---------------- phase 2: Ldt tile into shared memory (all threads) -----
        ptx::tc_fence_after_sync();
        const int ncols = jn / 2;
        for (int col = half * ncols; col < (half + 1) * ncols; col += 16) {
            float v[16];
            ptx::tmem_ld16(tmem + lane_off + col, v);
            float o[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int j = col + k;
                o[k] = (j <= i && j < len) ? v[k] * __expf(ai - sAcum[j]) * sDt[j] : 0.f;
            }
            const int kblk = col >> 6;
            const int ch = (col & 63) >> 3;
            uint8_t *row = sL + kblk * 2 * kRowBlock + (i_loc >> 3) * 1024 + (i_loc & 7) * 128;
            *reinterpret_cast<uint4 *>(row + ((ch ^ (i_loc & 7)) << 4)) =
                make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]),
                           pack_bf16(o[6], o[7]));
            *reinterpret_cast<uint4 *>(row + (((ch + 1) ^ (i_loc & 7)) << 4)) =
                make_uint4(pack_bf16(o[8], o[9]), pack_bf16(o[10], o[11]),
                           pack_bf16(o[12], o[13]), pack_bf16(o[14], o[15]));
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();

        // ---------------- phase 3: Ydiag = Ldt X (one thread) ---------------------
        if (tid == 0) {
            bool ok = ptx::mbar_wait(bar_x, 0, kWaitTimeoutNs);
            if (ok) {
                ptx::tc_fence_after_sync();
                const uint32_t id_d = ptx::idesc_bf16_f32(128, P_pad, 0, 1);
                const uint32_t aL = ptx::smem_u32(sL), aX = ptx::smem_u32(sX);
                for (int ks = 0; ks < jn / 16; ++ks) {
                    const uint64_t da =
                        ptx::sdesc_sw128(aL + (ks >> 2) * 2 * kRowBlock + (ks & 3) * 32, 16, 1024);
                    const uint64_t dx = ptx::sdesc_sw128(aX + ks * 2048, jn * 128, 1024);
                    ptx::mma_bf16_ss(tmem + kColOff + P_pad, da, dx, id_d, ks != 0);
                }
                ptx::mma_commit(bar_m);
                ok = ptx::mbar_wait(bar_m, nkb & 1, kWaitTimeoutNs);
            }
            if (!ok)
                *s_abort = 1;
        }
        __syncthreads();
    }

    if (!*s_abort) {
        // ---------------- epilogue: y = Ydiag + exp(Acum_i) Yoff + D x -----------
        ptx::tc_fence_after_sync();
        const float eai = __expf(ai);
        const float Dh = p.D ? p.D[h] : 0.f;
        const int ncols = P_pad / 2;
        const int64_t row_off = (static_cast<int64_t>(t0 + i) * p.H + h) * p.P;
        for (int col = half * ncols; col < (half + 1) * ncols; col += 16) {
            float yd[16], yo[16];
            ptx::tmem_ld16(tmem + lane_off + kColOff + P_pad + col, yd);
            ptx::tmem_ld16(tmem + lane_off + kColOff + col, yo);
            if (i < len && col < p.P) {
                const uint4 *xs = reinterpret_cast<const uint4 *>(p.x + row_off + col);
                uint4 xr[2] = {xs[0], xs[1]};
                const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(xr);
                uint32_t out[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float y0 = yd[2 * k] + eai * yo[2 * k] + Dh * __bfloat162float(xb[2 * k]);
                    const float y1 =
                        yd[2 * k + 1] + eai * yo[2 * k + 1] + Dh * __bfloat162float(xb[2 * k + 1]);
                    out[k] = pack_bf16(y0, y1);
                }
                uint4 *ys = reinterpret_cast<uint4 *>(p.y + row_off + col);
                ys[0] = make_uint4(out[0], out[1], out[2], out[3]);
                ys[1] = make_uint4(out[4], out[5], out[6], out[7]);
            }
        }
    } else if (tid == 0) {
        record_error(p.hdr, kErrTimeout);
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

SmemOptIn s_smem_configured;

}  // namespace

size_t chunk_scan_smem_bytes(const ScanParams &p)
{
    return k3_layout(pad64(p.P), pad64(p.N), p.Q).total + 1024;
}

cudaError_t launch_chunk_scan(const ScanParams &p, const ChunkScanMaps &maps,
                              cudaStream_t stream)
{
    const int P_pad = pad64(p.P), N_pad = pad64(p.N);
    const int n_itiles = (p.Q + 127) / 128;
    const size_t smem = chunk_scan_smem_bytes(p);
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void *>(chunk_scan_kernel), s_smem_configured);
    if (e != cudaSuccess)
        return e;
    dim3 grid(p.max_chunks * n_itiles, p.H);
    chunk_scan_kernel<<<grid, kThreads, smem, stream>>>(maps.C, maps.B, maps.X, maps.Sprev, p,
                                                        P_pad, N_pad, n_itiles);
    return cudaGetLastError();
}

}  // namespace ssd
