// Stages 2a, 2b and 4: per (block, group of heads)
//
//   CB[i,j]   = C_i . B_j                                       (tensor cores)
//   Ldt[i,j]  = CB[i,j] exp(Acum_i - Acum_j) dt_j   for j <= i, else 0
//   Ydiag     = Ldt X                                           (tensor cores)
//   Yoff      = C S_prev^T                                      (tensor cores)
//   y_i       = Ydiag_i + exp(Acum_i) Yoff_i + D[h] x_i         (bf16 out)
//
// These are the intra-chunk "attention-like" diagonal block built from
// segment sums, and the off-diagonal contribution of the state entering the
// block, of the kernelindex page "Mamba chunk scan with segsum"; the D skip is
// the last term of the "Per-token recurrence" of the Modular page
// "mamba2_ssd_scan".  A block is at most 128 tokens of one sequence (one MMA
// tile of rows); CB is computed once per block and shared by the CTA's heads.
//
// Warp roles (one CTA, 18 warps), heads processed as a pipeline:
//   warp 0    TMA producer: X of the first heads, C and B, then per head its
//             S_prev (after the state-passing kernel) and the next head's X
//   warp 1    tcgen05 issuer: CB once; per head Ydiag = Ldt X and Yoff = C S_prev^T
//             into a TMEM accumulator slot
//   warps 2-17 dt and cumulative decay; per head the masked Ldt tile (CB read
//             from TMEM, written to shared memory as a bf16 operand) and the
//             epilogue of the previous head (overlapping the MMAs of this one)
// C stays resident for every head's Yoff; S_prev tiles reuse B's space once
// CB is done.  Everything before the S_prev loads is independent of the
// state-passing kernel, so it overlaps that kernel (programmatic launch).
//
// The mask exp(Acum_i - Acum_j) is formed from differences of cumulative sums
// and never overflows for A <= 0: inside a 16-column chunk that lies wholly
// below row i it is the product exp(Acum_i - Acum_c) exp(Acum_c - Acum_j) with
// c the chunk's last column (both factors <= 1, the second shared by all
// rows); only the chunk holding the diagonal takes one exponential per element.
#include "kernels.cuh"
#include "sm100_ptx.cuh"
#include "ssd_device.cuh"
#include "trace.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 576;
constexpr int kMathThreads = 512;     // warps 2..17
constexpr int kMathWarps = 16;
constexpr int kRows = 128;
constexpr int kBlk16 = kRows * 128;   // 128 rows x 128 B swizzled block (16 KB)
constexpr int kNumBars = 16;
constexpr uint32_t kTmemCols = 512;

// Barrier indices.
enum {
    kCBFull = 0, kCBDone = 1, kXFull = 2, kXEmpty = 4, kSFull = 6, kSEmpty = 8,
    kLFull = 10, kLEmpty = 11, kYFull = 12, kYEmpty = 14
};

struct K3Layout {
    uint32_t sC, sBS, s_slot, sX, x_slot, sL, sDt, sAcum, sG, scratch, bars, tmem_slot, total;
};

// sC  : 128 rows (i) x N_pad, K-major, N_pad/64 blocks of 16 KB (resident)
// sBS : B (128 rows (j) x N_pad, K-major) for CB; afterwards nS slots of one
//       head's S_prev (P_pad rows x N_pad, K-major)
// sX  : nX slots of one head's X columns (128 rows x P_pad, MN-major)
// sL  : the 128 x 128 masked tile (K-major, 2 blocks of 16 KB)
__host__ __device__ inline K3Layout k3_layout(int P_pad, int N_pad, int HB, int nS, int nX)
{
    K3Layout L;
    const int nkb = N_pad / 64;
    const uint32_t bbytes = nkb * kBlk16;
    L.s_slot = nkb * P_pad * 128;
    L.x_slot = (P_pad / 64) * kBlk16;
    uint32_t off = 0;
    L.sC = off;
    off += nkb * kBlk16;
    L.sBS = off;
    off += bbytes > nS * L.s_slot ? bbytes : nS * L.s_slot;
    L.sX = off;
    off += nX * L.x_slot;
    L.sL = off;
    off += 2 * kBlk16;
    L.sDt = off;
    off += HB * kRows * 4;
    L.sAcum = off;
    off += HB * kRows * 4;
    L.sG = off;
    off += HB * kRows * 4;
    L.scratch = off;
    off += 64 * 4;
    L.bars = (off + 7) & ~7u;
    off = L.bars + kNumBars * 8;
    L.tmem_slot = off;
    off += 16;
    L.total = off;
    return L;
}

__device__ __forceinline__ void math_barrier()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kMathThreads) : "memory");
}

__global__ void __launch_bounds__(kThreads)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmS, ScanParams p, K3Config cfg)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int HB = cfg.HB, P_pad = cfg.P_pad, N_pad = cfg.N_pad, nS = cfg.nS, nX = cfg.nX,
              nY = cfg.nY;
    const K3Layout L = k3_layout(P_pad, N_pad, HB, nS, nX);
    uint8_t *sC = smem + L.sC;
    uint8_t *sBS = smem + L.sBS;
    uint8_t *sX = smem + L.sX;
    uint8_t *sL = smem + L.sL;
    float *sDt = reinterpret_cast<float *>(smem + L.sDt);
    float *sAcum = reinterpret_cast<float *>(smem + L.sAcum);
    float *sG = reinterpret_cast<float *>(smem + L.sG);
    int32_t *scratch = reinterpret_cast<int32_t *>(smem + L.scratch);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.tmem_slot + 4);
    float *s_part = reinterpret_cast<float *>(scratch + 40);

    const int blk = blockIdx.x;
    const int h0 = blockIdx.y * HB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0)
        SSD_TRACE_EV(2, 0);

    const BlockInfo bi = map_block<kThreads>(p, blk, scratch, nullptr);
    if (!bi.valid || bi.seq < 0)
        return;
    const int t0 = bi.t0, len = bi.len;
    const int g = h0 / (p.H / p.G);
    const int nkb = N_pad / 64;
    const uint32_t slot_idx = p.cache_idx[bi.seq];
    // the state entering the block is zero for a first block without initial state
    const bool has_prev = !bi.first || (p.has_init != nullptr && p.has_init[bi.seq] != 0 &&
                                        static_cast<int64_t>(slot_idx) < p.max_slots);

    if (tid == 0) {
        for (int k = 0; k < kNumBars; ++k) {
            const bool math_arrivals = k == kLFull || k == kXEmpty || k == kXEmpty + 1 ||
                                       k == kYEmpty || k == kYEmpty + 1;
            ptx::mbar_init(bars + k, math_arrivals ? kMathWarps : 1);
        }
        ptx::fence_barrier_init();
        *s_abort = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0)
        SSD_TRACE_EV(2, 1);
    // TMEM columns: CB [0,128); accumulator slot ys: Ydiag at 128 + ys*2*P_pad, Yoff after it
    auto col_yd = [&](int ys) { return 128u + static_cast<uint32_t>(ys * 2 * P_pad); };
    auto col_yo = [&](int ys) { return 128u + static_cast<uint32_t>(ys * 2 * P_pad + P_pad); };
    // first column of the 64-wide blocks that hold head (h0+hh)'s x
    auto x_col0 = [&](int hh) { return ((h0 + hh) * p.P / 64) * 64; };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            auto load_x = [&](int hh) {
                const int xs = hh % nX;
                uint8_t *dst = sX + xs * L.x_slot;
                ptx::mbar_arrive_expect_tx(bars + kXFull + xs, L.x_slot);
                for (int cb = 0; cb < P_pad / 64; ++cb)
                    for (int rb = 0; rb < 2; ++rb)
                        ptx::tma_load_3d(dst + cb * kBlk16 + rb * 8192, &tmX, bars + kXFull + xs,
                                         x_col0(hh) + cb * 64, t0 + rb * 64, 0);
            };
            for (int hh = 0; hh < nX && hh < HB; ++hh)
                load_x(hh);
            ptx::mbar_arrive_expect_tx(bars + kCBFull, 2 * nkb * kBlk16);
            for (int kb = 0; kb < nkb; ++kb)
                for (int rb = 0; rb < 2; ++rb) {
                    ptx::tma_load_3d(sC + kb * kBlk16 + rb * 8192, &tmC, bars + kCBFull, kb * 64, g,
                                     t0 + rb * 64);
                    ptx::tma_load_3d(sBS + kb * kBlk16 + rb * 8192, &tmB, bars + kCBFull, kb * 64,
                                     g, t0 + rb * 64);
                }
            SSD_TRACE_EV(2, 2);
            if (has_prev) {
                pdl_wait();
                SSD_TRACE_EV(2, 3);
            }
            // per head: its S_prev (slot freed by the Yoff MMAs nS heads back, or by
            // CB for a slot's first use since S_prev overlays B), then its X when
            // the ring did not hold it yet (slot freed by the epilogue nX heads back)
            for (int hh = 0; hh < HB && ok; ++hh) {
                if (has_prev) {
                    const int ss = hh % nS, use = hh / nS;
                    const bool free_slot =
                        use == 0 ? ptx::mbar_wait(bars + kCBDone, 0, kWaitTimeoutNs)
                                 : ptx::mbar_wait(bars + kSEmpty + ss, (use - 1) & 1, kWaitTimeoutNs);
                    if (!free_slot || *s_abort) {
                        ok = false;
                        break;
                    }
                    uint8_t *dst = sBS + ss * L.s_slot;
                    if (hh == 0)
                        SSD_TRACE_EV(2, 24);
                    ptx::mbar_arrive_expect_tx(bars + kSFull + ss, L.s_slot);
                    for (int kb = 0; kb < nkb; ++kb)
                        for (int pb = 0; pb < P_pad / 64; ++pb)
                            ptx::tma_load_3d(dst + kb * P_pad * 128 + pb * 8192, &tmS,
                                             bars + kSFull + ss, kb * 64, pb * 64,
                                             blk * p.H + h0 + hh);
                }
                if (hh >= nX) {
                    const int xs = hh % nX, use = hh / nX;
                    if (!ptx::mbar_wait(bars + kXEmpty + xs, (use - 1) & 1, kWaitTimeoutNs) ||
                        *s_abort) {
                        ok = false;
                        break;
                    }
                    load_x(hh);
                }
            }
            SSD_TRACE_EV(2, 4);
            if (!ok)
                *s_abort = 1;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = ptx::mbar_wait(bars + kCBFull, 0, kWaitTimeoutNs);
            if (ok) {
                ptx::tc_fence_after_sync();
                const uint32_t id_cb = ptx::idesc_bf16_f32(128, 128, 0, 0);
                const uint64_t dC0 = ptx::sdesc_sw128(ptx::smem_u32(sC), 16, 1024);
                const uint64_t dB0 = ptx::sdesc_sw128(ptx::smem_u32(sBS), 16, 1024);
                for (int kb = 0; kb < nkb; ++kb) {
                    const uint64_t dC = ptx::sdesc_add(dC0, kb * kBlk16);
                    const uint64_t dB = ptx::sdesc_add(dB0, kb * kBlk16);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        ptx::mma_bf16_ss(tmem, ptx::sdesc_add(dC, ks * 32), ptx::sdesc_add(dB, ks * 32),
                                         id_cb, (kb | ks) != 0);
                }
                ptx::mma_commit(bars + kCBDone);
            }
            SSD_TRACE_EV(2, 5);
            const uint32_t id_d = ptx::idesc_bf16_f32(128, P_pad, 0, 1);
            const uint32_t id_o = ptx::idesc_bf16_f32(128, P_pad, 0, 0);
            const uint64_t dL0 = ptx::sdesc_sw128(ptx::smem_u32(sL), 16, 1024);
            const uint64_t dX0 = ptx::sdesc_sw128(ptx::smem_u32(sX), kBlk16, 1024);
            const uint64_t dCk = ptx::sdesc_sw128(ptx::smem_u32(sC), 16, 1024);
            const uint64_t dS0 = ptx::sdesc_sw128(ptx::smem_u32(sBS), 16, 1024);
            const int nks = (len + 15) / 16;
            for (int hh = 0; hh < HB && ok; ++hh) {
                const int ys = hh % nY, uy = hh / nY, xs = hh % nX, ss = hh % nS;
                ok = (uy == 0 || ptx::mbar_wait(bars + kYEmpty + ys, (uy - 1) & 1, kWaitTimeoutNs)) &&
                     ptx::mbar_wait(bars + kXFull + xs, (hh / nX) & 1, kWaitTimeoutNs) &&
                     ptx::mbar_wait(bars + kLFull, hh & 1, kWaitTimeoutNs) && !*s_abort;
                if (!ok)
                    break;
                if (hh == 0)
                    SSD_TRACE_EV(2, 25);
                ptx::tc_fence_after_sync();
                const uint64_t dX = ptx::sdesc_add(dX0, xs * L.x_slot);
                for (int ks = 0; ks < nks; ++ks)
                    ptx::mma_bf16_ss(tmem + col_yd(ys),
                                     ptx::sdesc_add(dL0, (ks >> 2) * kBlk16 + (ks & 3) * 32),
                                     ptx::sdesc_add(dX, ks * 2048), id_d, ks != 0);
                if (hh == 0)
                    SSD_TRACE_EV(2, 27);
                ptx::mma_commit(bars + kLEmpty);
                if (has_prev) {
                    if (!ptx::mbar_wait(bars + kSFull + ss, (hh / nS) & 1, kWaitTimeoutNs)) {
                        ok = false;
                        break;
                    }
                    if (hh == 0)
                        SSD_TRACE_EV(2, 26);
                    ptx::tc_fence_after_sync();
                    const uint64_t dS = ptx::sdesc_add(dS0, ss * L.s_slot);
                    for (int kb = 0; kb < nkb; ++kb) {
                        const uint64_t dCb = ptx::sdesc_add(dCk, kb * kBlk16);
                        const uint64_t dSb = ptx::sdesc_add(dS, kb * P_pad * 128);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            ptx::mma_bf16_ss(tmem + col_yo(ys), ptx::sdesc_add(dCb, ks * 32),
                                             ptx::sdesc_add(dSb, ks * 32), id_o, (kb | ks) != 0);
                    }
                    if (hh == 0)
                        SSD_TRACE_EV(2, 28);
                    ptx::mma_commit(bars + kSEmpty + ss);
                }
                ptx::mma_commit(bars + kYFull + ys);
                SSD_TRACE_EV(2, 6 + (hh < 3 ? hh : 3));
            }
            if (!ok)
                *s_abort = 1;
            SSD_TRACE_EV(2, 10);
        }
    } else {
        // ------------------------------------------------------------ math warps
        const int mt = tid - 64;             // 0..511
        const int mw = warp - 2;             // math warp 0..15
        const int quarter = mt >> 7, jj = mt & 127;
        // dt of every head of the CTA at once (one round trip), then the scans
        float dv[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int hh = 4 * k + quarter;
            dv[k] = (hh < HB && jj < len) ? processed_dt(p, t0 + jj, h0 + hh) : 0.f;
        }
        if (mt == 0)
            SSD_TRACE_EV(2, 23);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (4 * k >= HB)
                break;
            const int hh = 4 * k + quarter;
            const float a = hh < HB ? p.A[h0 + hh] * dv[k] : 0.f;
            const float incl = warp_inclusive_scan(a);
            if (lane == 31)
                s_part[mw] = incl;
            math_barrier();
            float before = 0.f;
            for (int w = quarter * 4; w < mw; ++w)
                before += s_part[w];
            if (hh < HB) {
                sDt[hh * kRows + jj] = dv[k];
                sAcum[hh * kRows + jj] = before + incl;
            }
            math_barrier();
        }
        for (int k = mt; k < HB * kRows; k += kMathThreads) {
            const int hh = k / kRows, j = k % kRows;
            // exp(Acum_c - Acum_j) dt_j with c the last column of j's 16-column chunk
            sG[k] = __expf(sAcum[hh * kRows + (j | 15)] - sAcum[k]) * sDt[k];
        }
        math_barrier();
        if (mt == 0)
            SSD_TRACE_EV(2, 11);

        const int q = warp & 3;
        const int i = q * 32 + lane;          // block-local row of this thread
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const int col_base = quarter * 32;    // this thread's 32 CB columns
        bool ok = ptx::mbar_wait(bars + kCBDone, 0, kWaitTimeoutNs);
        if (mt == 0)
            SSD_TRACE_EV(2, 12);

        auto epilogue = [&](int hh) -> bool {
            const int ys = hh % nY, xs = hh % nX;
            if (!ptx::mbar_wait(bars + kYFull + ys, (hh / nY) & 1, kWaitTimeoutNs) ||
                !ptx::mbar_wait(bars + kXFull + xs, (hh / nX) & 1, kWaitTimeoutNs))
                return false;
            ptx::tc_fence_after_sync();
            if (mt == 0 && hh == 0)
                SSD_TRACE_EV(2, 21);
            const float eai = has_prev ? __expf(sAcum[hh * kRows + i]) : 0.f;
            const float Dh = p.D ? p.D[h0 + hh] : 0.f;
            const int xoff = (h0 + hh) * p.P - x_col0(hh);   // head's first column in its X slot
            const uint8_t *xsl = sX + xs * L.x_slot;
            const int ncols = P_pad / 4;
#pragma unroll 1
            for (int col = quarter * ncols; col < (quarter + 1) * ncols; col += 16) {
                if (col >= p.P)
                    break;
                float yd[16], yo[16];
                // head hh's columns start at xoff inside its 64-wide X block
                ptx::tmem_ld16(tmem + lane_off + col_yd(ys) + xoff + col, yd);
                if (has_prev)
                    ptx::tmem_ld16(tmem + lane_off + col_yo(ys) + col, yo);
                if (i < len) {
                    const int xc = xoff + col;
                    const uint8_t *xrow = xsl + (xc >> 6) * kBlk16 + (i >> 3) * 1024 + (i & 7) * 128;
                    const int ch = (xc & 63) >> 3;
                    uint4 xr[2];
                    xr[0] = *reinterpret_cast<const uint4 *>(xrow + ((ch ^ (i & 7)) << 4));
                    xr[1] = *reinterpret_cast<const uint4 *>(xrow + (((ch + 1) ^ (i & 7)) << 4));
                    const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(xr);
                    uint32_t out[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        float y0 = yd[2 * k] + Dh * __bfloat162float(xb[2 * k]);
                        float y1 = yd[2 * k + 1] + Dh * __bfloat162float(xb[2 * k + 1]);
                        if (has_prev) {
                            y0 += eai * yo[2 * k];
                            y1 += eai * yo[2 * k + 1];
                        }
                        out[k] = pack_bf16(y0, y1);
                    }
                    uint4 *ys_ptr = reinterpret_cast<uint4 *>(
                        p.y + (static_cast<int64_t>(t0 + i) * p.H + h0 + hh) * p.P + col);
                    ys_ptr[0] = make_uint4(out[0], out[1], out[2], out[3]);
                    ys_ptr[1] = make_uint4(out[4], out[5], out[6], out[7]);
                }
            }
            if (mt == 0 && hh == 0)
                SSD_TRACE_EV(2, 22);
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(bars + kYEmpty + ys);
                ptx::mbar_arrive(bars + kXEmpty + xs);
            }
            return true;
        };

        for (int hh = 0; hh <= HB && ok; ++hh) {
            if (hh < HB) {
                if (hh >= 1 && !ptx::mbar_wait(bars + kLEmpty, (hh - 1) & 1, kWaitTimeoutNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const float *acum = sAcum + hh * kRows;
                const float *dtv = sDt + hh * kRows;
                const float *gv = sG + hh * kRows;
                const float ai = acum[i];
                // one 16-column chunk per iteration; the loop stays rolled so that
                // the math warps' code does not crowd the MMA issuer's out of the
                // instruction cache they share
#pragma unroll 1
                for (int c16 = 0; c16 < 2; ++c16) {
                    const int col = col_base + c16 * 16;
                    float v[16];
                    ptx::tmem_ld16(tmem + lane_off + col, v);
                    if (mt == 0 && hh == 0 && c16 == 0)
                        SSD_TRACE_EV(2, 19);
                    float o[16];
                    if (col + 15 < i) {
                        const float e = __expf(ai - acum[col + 15]);
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            o[k] = v[k] * e * gv[col + k];
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const int j = col + k;
                            o[k] = j <= i ? v[k] * __expf(ai - acum[j]) * dtv[j] : 0.f;
                        }
                    }
                    uint8_t *row = sL + (col >> 6) * kBlk16 + (i >> 3) * 1024 + (i & 7) * 128;
                    const int ch = (col & 63) >> 3;
                    *reinterpret_cast<uint4 *>(row + ((ch ^ (i & 7)) << 4)) =
                        make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]),
                                   pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
                    *reinterpret_cast<uint4 *>(row + (((ch + 1) ^ (i & 7)) << 4)) =
                        make_uint4(pack_bf16(o[8], o[9]), pack_bf16(o[10], o[11]),
                                   pack_bf16(o[12], o[13]), pack_bf16(o[14], o[15]));
                }
                if (mt == 0 && hh == 0)
                    SSD_TRACE_EV(2, 20);
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(bars + kLFull);
                if (mt == 0)
                    SSD_TRACE_EV(2, 13 + (hh < 3 ? hh : 3));
            }
            if (hh >= 1 && !epilogue(hh - 1)) {
                ok = false;
                break;
            }
        }
        if (mt == 0)
            SSD_TRACE_EV(2, 17);
        if (!ok)
            *s_abort = 1;
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0)
        SSD_TRACE_EV(2, 18);
    if (tid == 0 && *s_abort)
        record_error(p.hdr, kErrTimeout);
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

SmemOptIn s_smem_configured;

}  // namespace

K3Config chunk_scan_config(int H, int G, int P, int N)
{
    K3Config c{};
    const int hpg = H / G;
    c.P_pad = pad64(P);
    c.N_pad = pad64(N);
    c.nY = (512 - 128) / (2 * c.P_pad);
    if (c.nY > 2)
        c.nY = 2;
    // heads per CTA: the largest divisor of the group's heads up to 4 (the
    // heads share one CB; the dt prologue holds at most 8)
    for (int hb = hpg < 4 ? hpg : 4; hb >= 1; --hb) {
        if (hpg % hb)
            continue;
        c.HB = hb;
        break;
    }
    // ring depths: two S_prev / X slots when they fit the shared-memory budget
    for (int nS = 2; nS >= 1; --nS) {
        for (int nX = 2; nX >= 1; --nX) {
            const size_t smem = k3_layout(c.P_pad, c.N_pad, c.HB, nS, nX).total + 1024;
            if (smem <= static_cast<size_t>(kMaxSmemPerBlock)) {
                c.nS = nS;
                c.nX = nX;
                c.smem = smem;
                return c;
            }
        }
    }
    c.HB = 0;  // does not fit
    return c;
}

cudaError_t launch_chunk_scan(const ScanParams &p, const ChunkScanMaps &maps, cudaStream_t stream,
                              bool programmatic)
{
    const K3Config c = chunk_scan_config(p.H, p.G, p.P, p.N);
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void *>(chunk_scan_kernel), s_smem_configured);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.max_chunks, p.H / c.HB);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chunk_scan_kernel, maps.C, maps.B, maps.X, maps.Sprev, p, c);
}

}  // namespace ssd
