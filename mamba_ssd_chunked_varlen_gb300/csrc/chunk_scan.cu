// Stages 2a, 2b and 4: per (block, group of heads)
//
//   CB[i,j]   = C_i . B_j                                       (tensor cores)
//   Ldt[i,j]  = CB[i,j] exp(Acum_i - Acum_j) dt_j   for j <= i, else 0
//   Ydiag     = (Ldt + D[h] I) X                                (tensor cores)
//   Yoff      = C S_prev^T                                      (tensor cores)
//   y_i       = Ydiag_i + exp(Acum_i) Yoff_i                    (bf16 out)
//
// These are the intra-chunk "attention-like" diagonal block built from
// segment sums, and the off-diagonal contribution of the state entering the
// block, of the kernelindex page "Mamba chunk scan with segsum"; the D skip is
// the last term of the "Per-token recurrence" of the Modular page
// "mamba2_ssd_scan", folded into the diagonal of the masked tile so that it
// rides along with the diagonal MMA.  A block is at most 128 tokens of one
// sequence (one MMA tile of rows); CB is computed once per block and shared by
// the CTA's heads.
//
// The heads form off-diagonal groups of up to two (their S_prev tiles stacked
// along N of one MMA, C shared).  Warp roles (one CTA, 18 warps):
//   warp 0    TMA producer: X of the CTA's heads, C and B; after the
//             previous kernel (state passing, or the fused walk), each
//             group's S_prev tiles into B's space
//             (free once CB, then the previous group's Yoff, is done)
//   warp 1    tcgen05 issuer: CB; group by group, Ydiag = Ldt X per head with
//             the masked tile read from tensor memory, then the group's
//             Yoff = C [S_prev_h ...]^T
//   warps 2-17 dt and cumulative decay; CB read once from tensor memory into
//             registers; per head the masked tile, written back to tensor
//             memory as the bf16 A operand (two slots, so that building one
//             head's tile overlaps the MMA of the previous one); then the
//             epilogue group by group, y staged through shared memory so that
//             every warp store writes whole 128-byte rows
// Everything before the S_prev loads is independent of the previous kernel,
// so it may overlap that kernel's tail (programmatic launch).
//
// Tensor memory (512 columns): [0,128) CB, then the two masked-tile slots
// (64 columns each, bf16 pairs); [128,384) Ydiag of up to four heads;
// [384,512) the Yoff accumulator of the current group.
//
// The mask exp(Acum_i - Acum_j) is formed from differences of cumulative sums
// and factored per 16-column chunk so that a row takes one exponential per
// chunk: for a chunk wholly below row i it is exp(Acum_i - Acum_c) exp(Acum_c -
// Acum_j) with c the chunk's last column (both factors <= 1 for A <= 0, the
// second shared by all rows); for the chunk holding the diagonal the reference
// is the chunk's first column, which keeps both factors within e^+-40 when the
// chunk's own decay spans at most e^40 -- otherwise that chunk takes one
// exponential per element.
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
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColYd = 128;      // Ydiag of head hh at kColYd + hh * P_pad
constexpr uint32_t kColYo = 384;      // Yoff accumulator of the current group

// Barrier indices.
enum {
    kCBFull = 0,   // C and B landed
    kXFull = 1,    // X landed
    kCBDone = 2,   // CB accumulator final (B's space free)
    kLFull = 3,    // [2] masked-tile slot written (one arrival per math warp)
    kLEmpty = 5,   // [2] masked-tile slot read by its MMAs
    kYoEmpty = 7,  // Yoff accumulator drained by the epilogue (one arrival per math warp)
    kSFull = 8,    // [2] S_prev tiles of an off-diagonal group landed
    kYoFull = 10,  // [2] accumulators of an off-diagonal group final (B's space free)
    kDrain = 12,   // every MMA of the CTA done (before tensor memory is freed)
    kNumBars = 13
};

struct K3Layout {
    uint32_t sC, sB, sX, sY, sDt, sAcum, sG, scratch, bars, tmem_slot, total;
};

// sC : 128 rows (i) x N_pad, K-major, N_pad/64 blocks of 16 KB (resident)
// sB : B (128 rows (j) x N_pad, K-major) for CB; afterwards each group's
//      S_prev tiles in turn (YG*P_pad rows x N_pad, K-major)
// sX : n_xb 64-column blocks of X (128 rows x 64, MN-major)
// sY : one 128 x 64 bf16 tile of y on its way out (rows of 128 B, 16-byte
//      chunks XOR-swizzled by row)
__host__ __device__ inline K3Layout k3_layout(int N_pad, int HB, int n_xb)
{
    K3Layout L;
    const int nkb = N_pad / 64;
    uint32_t off = 0;
    L.sC = off;
    off += nkb * kBlk16;
    L.sB = off;
    off += nkb * kBlk16;
    L.sX = off;
    off += n_xb * kBlk16;
    L.sY = off;
    off += kBlk16;
    L.sDt = off;
    off += HB * kRows * 4;
    L.sAcum = off;
    off += HB * kRows * 4;
    L.sG = off;
    off += 2 * HB * kRows * 4 + 16 + HB * 8 * 4;   // gv, hv (offset by 16 B), safe flags
    L.scratch = off;
    off += 64 * 4;   // block map (36 ints), warp partials (16), D (8)
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

// Barrier over the math warps that also returns whether any of them passed true
// (keeps loop exits uniform, so that no math warp is left waiting at a barrier).
__device__ __forceinline__ bool math_barrier_any(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(kMathThreads)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmS, ScanParams p, K3Config cfg)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int HB = cfg.HB, P_pad = cfg.P_pad, N_pad = cfg.N_pad, YG = cfg.YG;
    const int n_groups = (HB + YG - 1) / YG;
    const K3Layout L = k3_layout(N_pad, HB, cfg.n_xb);
    uint8_t *sC = smem + L.sC;
    uint8_t *sB = smem + L.sB;
    uint8_t *sX = smem + L.sX;
    uint8_t *sY = smem + L.sY;
    float *sDt = reinterpret_cast<float *>(smem + L.sDt);
    float *sAcum = reinterpret_cast<float *>(smem + L.sAcum);
    float *sG = reinterpret_cast<float *>(smem + L.sG);                 // [HB][128]
    float *sH = sG + HB * kRows + 4;                                      // [HB][128]
    int32_t *sSafe = reinterpret_cast<int32_t *>(sH + HB * kRows);        // [HB][8]
    int32_t *scratch = reinterpret_cast<int32_t *>(smem + L.scratch);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.tmem_slot + 4);
    float *s_part = reinterpret_cast<float *>(scratch + 40);   // 16 warp partials
    float *sD = reinterpret_cast<float *>(scratch + 56);       // D of the CTA's heads (<= 8)

    const bool by_rows = blocks_on_y(p);
    const int blk = by_rows ? blockIdx.y : blockIdx.x;
    const int h0 = (by_rows ? blockIdx.x : blockIdx.y) * HB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0)
        SSD_TRACE_EV(2, 0);

    if (tid == 0) {
        ptx::prefetch_tensormap(&tmC);
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmX);
        ptx::prefetch_tensormap(&tmS);
    }
    // with the block table the block-map kernel has completed (the chunk-state
    // CTAs read it before letting later kernels launch)
    const BlockInfo bi = p.table != nullptr ? lookup_block(p, blk)
                                            : map_block<kThreads>(p, blk, scratch, nullptr);
    // Every CTA waits for the previous grid before it leaves (those without an
    // entering state would not otherwise), so that this grid completes only
    // after its predecessors and a dependent launch may rely on all of them.
    if (!bi.valid || bi.seq < 0) {
        pdl_wait();
        return;
    }
    const int t0 = bi.t0, len = bi.len;
    const int g = h0 / (p.H / p.G);
    const int nkb = N_pad / 64;
    // the state entering the block is zero for a first block without initial state
    const bool has_prev = !bi.first || seq_init_index(p, bi.seq) >= 0;
    // X columns of the CTA's heads, loaded from a 64-aligned start
    const int x_base = (h0 * p.P / 64) * 64;
    const int n_xb = ((h0 + HB) * p.P - x_base + 63) / 64;

    if (tid == 0) {
        for (int k = 0; k < kNumBars; ++k)
            ptx::mbar_init(bars + k, (k == kLFull || k == kLFull + 1 || k == kYoEmpty) ? kMathWarps : 1);
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
    // Yoff group gi: heads [gi*YG, min(HB, (gi+1)*YG)), N = heads * P_pad
    auto group_n = [&](int gi) { return (HB - gi * YG < YG ? HB - gi * YG : YG) * P_pad; };
    auto group_end = [&](int gi) { return (gi + 1) * YG < HB ? (gi + 1) * YG : HB; };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            ptx::mbar_arrive_expect_tx(bars + kXFull, n_xb * kBlk16);
            for (int xb = 0; xb < n_xb; ++xb)
                for (int rb = 0; rb < 2; ++rb)
                    ptx::tma_load_3d(sX + xb * kBlk16 + rb * 8192, &tmX, bars + kXFull,
                                     x_base + xb * 64, t0 + rb * 64, 0);
            ptx::mbar_arrive_expect_tx(bars + kCBFull, 2 * nkb * kBlk16);
            for (int kb = 0; kb < nkb; ++kb)
                for (int rb = 0; rb < 2; ++rb) {
                    ptx::tma_load_3d(sC + kb * kBlk16 + rb * 8192, &tmC, bars + kCBFull, kb * 64, g,
                                     t0 + rb * 64);
                    ptx::tma_load_3d(sB + kb * kBlk16 + rb * 8192, &tmB, bars + kCBFull, kb * 64,
                                     g, t0 + rb * 64);
                }
            SSD_TRACE_EV(2, 2);
            int armed = 0;   // S_prev groups whose loads were issued
            if (has_prev) {
                pdl_wait();
                SSD_TRACE_EV(2, 3);
                for (int gi = 0; gi < n_groups && ok; ++gi) {
                    // B's space is free once CB is done, then once the previous
                    // group's Yoff MMAs are done
                    ok = ptx::mbar_wait(bars + (gi == 0 ? kCBDone : kYoFull + gi - 1), 0,
                                        kWaitTimeoutNs) &&
                         !*s_abort;
                    if (!ok)
                        break;
                    const int gn = group_n(gi);
                    uint8_t *dst = sB;
                    ptx::mbar_arrive_expect_tx(bars + kSFull + gi, nkb * gn * 128);
                    for (int kb = 0; kb < nkb; ++kb)
                        for (int r = 0; r < gn; r += 64) {
                            const int hl = r / P_pad, pb = (r % P_pad) / 64;
                            ptx::tma_load_3d(dst + kb * gn * 128 + r * 128, &tmS, bars + kSFull + gi,
                                             kb * 64, pb * 64, blk * p.H + h0 + gi * YG + hl);
                        }
                    ++armed;
                }
                SSD_TRACE_EV(2, 4);
            }
            if (!ok)
                *s_abort = 1;
            // copies still in flight must land before the CTA exits
            ptx::mbar_wait(bars + kXFull, 0, kWaitTimeoutNs);
            ptx::mbar_wait(bars + kCBFull, 0, kWaitTimeoutNs);
            for (int gi = 0; gi < armed; ++gi)
                ptx::mbar_wait(bars + kSFull + gi, 0, kWaitTimeoutNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = ptx::mbar_wait(bars + kCBFull, 0, kWaitTimeoutNs);
            if (ok) {
                ptx::tc_fence_after_sync();
                const uint32_t id_cb = ptx::idesc_bf16_f32(128, 128, 0, 0);
                const uint64_t dC0 = ptx::sdesc_sw128(ptx::smem_u32(sC), 16, 1024);
                const uint64_t dB0 = ptx::sdesc_sw128(ptx::smem_u32(sB), 16, 1024);
                for (int kb = 0; kb < nkb; ++kb) {
                    const uint64_t dC = ptx::sdesc_add(dC0, kb * kBlk16);
                    const uint64_t dB = ptx::sdesc_add(dB0, kb * kBlk16);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        ptx::mma_bf16_ss(tmem, ptx::sdesc_add(dC, ks * 32), ptx::sdesc_add(dB, ks * 32),
                                         id_cb, (kb | ks) != 0);
                }
                ptx::mma_commit(bars + kCBDone);
                SSD_TRACE_EV(2, 5);
                ok = ptx::mbar_wait(bars + kXFull, 0, kWaitTimeoutNs);
                SSD_TRACE_EV(2, 29);
            }
            const uint32_t id_d = ptx::idesc_bf16_f32(128, P_pad, 0, 1);
            const uint64_t dX0 = ptx::sdesc_sw128(ptx::smem_u32(sX), kBlk16, 1024);
            const uint64_t dCk = ptx::sdesc_sw128(ptx::smem_u32(sC), 16, 1024);
            const uint64_t dS0 = ptx::sdesc_sw128(ptx::smem_u32(sB), 16, 1024);
            const int nks = (len + 15) / 16;
            for (int gi = 0; gi < n_groups && ok; ++gi) {
                // diagonal: one head at a time, A = its masked tile in tensor memory
                for (int hh = gi * YG; hh < group_end(gi) && ok; ++hh) {
                    const int ls = hh & 1;
                    ok = ptx::mbar_wait(bars + kLFull + ls, (hh >> 1) & 1, kWaitTimeoutNs) && !*s_abort;
                    if (!ok)
                        break;
                    ptx::tc_fence_after_sync();
                    const int xb = ((h0 + hh) * p.P - x_base) >> 6;
                    const uint64_t dX = ptx::sdesc_add(dX0, xb * kBlk16);
                    const uint32_t d = tmem + kColYd + hh * P_pad;
                    const uint32_t a = tmem + ls * 64;
                    for (int ks = 0; ks < nks; ++ks)
                        ptx::mma_bf16_ts(d, a + ks * 8, ptx::sdesc_add(dX, ks * 2048), id_d, ks != 0);
                    ptx::mma_commit(bars + kLEmpty + ls);
                    if (hh < 4)
                        SSD_TRACE_EV(2, 24 + hh);
                }
                // off-diagonal: A = C (shared), B = the group's S_prev tiles; the
                // accumulator is free once the previous group's epilogue drained it
                if (has_prev && ok) {
                    ok = ptx::mbar_wait(bars + kSFull + gi, 0, kWaitTimeoutNs) &&
                         (gi == 0 || ptx::mbar_wait(bars + kYoEmpty, (gi - 1) & 1, kWaitTimeoutNs)) &&
                         !*s_abort;
                    if (!ok)
                        break;
                    ptx::tc_fence_after_sync();
                    const int gn = group_n(gi);
                    const uint32_t id_o = ptx::idesc_bf16_f32(128, gn, 0, 0);
                    for (int kb = 0; kb < nkb; ++kb) {
                        const uint64_t dCb = ptx::sdesc_add(dCk, kb * kBlk16);
                        const uint64_t dSb = ptx::sdesc_add(dS0, kb * gn * 128);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            ptx::mma_bf16_ss(tmem + kColYo, ptx::sdesc_add(dCb, ks * 32),
                                             ptx::sdesc_add(dSb, ks * 32), id_o, (kb | ks) != 0);
                    }
                }
                ptx::mma_commit(bars + kYoFull + gi);
                SSD_TRACE_EV(2, 6 + gi);
            }
            SSD_TRACE_EV(2, 8);
            if (!ok)
                *s_abort = 1;
            // every MMA issued must finish before tensor memory is released
            ptx::mma_commit(bars + kDrain);
            ptx::mbar_wait(bars + kDrain, 0, kWaitTimeoutNs);
        }
    } else {
        // ------------------------------------------------------------ math warps
        const int mt = tid - 64;             // 0..511
        const int mw = warp - 2;             // math warp 0..15
        const int quarter = mt >> 7, jj = mt & 127;
        // dt of every head of the CTA at once (one round trip), then the scans
        float dv[2], av[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int hh = 4 * k + quarter;
            dv[k] = (hh < HB && jj < len) ? processed_dt(p, t0 + jj, h0 + hh) : 0.f;
            av[k] = hh < HB ? p.A[h0 + hh] : 0.f;
        }
        const float d_own = (mt < HB && p.D) ? p.D[h0 + mt] : 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (4 * k >= HB)
                break;
            const int hh = 4 * k + quarter;
            const float incl = warp_inclusive_scan(av[k] * dv[k]);
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
            const float *ac = sAcum + hh * kRows;
            // exp(Acum_r - Acum_j) dt_j with r the last (gv) or the first (hv)
            // column of j's 16-column chunk
            sG[k] = __expf(ac[j | 15] - ac[j]) * sDt[k];
            sH[k] = __expf(ac[j & ~15] - ac[j]) * sDt[k];
            // a chunk whose cumulative decay spans at most e^40 may factor its
            // diagonal tile around its first column without over- or underflow
            if ((j & 15) == 0)
                sSafe[hh * 8 + (j >> 4)] = fabsf(ac[j] - ac[j + 15]) <= 40.f;
        }
        if (mt < HB)
            sD[mt] = d_own;
        math_barrier();
        if (mt == 0)
            SSD_TRACE_EV(2, 9);

        const int q = warp & 3;
        const int i = q * 32 + lane;          // block-local row of this thread
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        // this thread's CB columns: the 16-column chunks `quarter` and
        // `quarter + 4`, so that every warp holds at most one chunk crossing
        // the diagonal of its rows
        const int col0 = quarter * 16, col1 = 64 + quarter * 16;
        bool ok = ptx::mbar_wait(bars + kCBDone, 0, kWaitTimeoutNs);
        ptx::tc_fence_after_sync();
        float cb[32];
        {
            float v[16];
            ptx::tmem_ld16(tmem + lane_off + col0, v);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                cb[k] = v[k];
            ptx::tmem_ld16(tmem + lane_off + col1, v);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                cb[16 + k] = v[k];
        }
        // every thread holds its CB values before the tile slots overwrite them
        ptx::tc_fence_before_sync();
        math_barrier();
        ptx::tc_fence_after_sync();
        if (mt == 0)
            SSD_TRACE_EV(2, 10);

        for (int hh = 0; hh < HB && ok; ++hh) {
            const int ls = hh & 1;
            if (hh >= 2) {
                ok = ptx::mbar_wait(bars + kLEmpty + ls, ((hh - 2) >> 1) & 1, kWaitTimeoutNs);
                if (!ok)
                    break;
                ptx::tc_fence_after_sync();
            }
            if (mt == 64 && hh < 4)
                SSD_TRACE_EV(2, 16 + 2 * hh);
            const float *acum = sAcum + hh * kRows;
            const float *dtv = sDt + hh * kRows;
            const float *gv = sG + hh * kRows;
            const float *hv = sH + hh * kRows;
            const float ai = acum[i];
            const float Dh = sD[hh];
            uint32_t packed[16];
#pragma unroll
            for (int c16 = 0; c16 < 2; ++c16) {
                const int col = c16 ? col1 : col0;
                const int lim = i - col;          // columns k <= lim lie at or below row i
                float o[16];
                if (col + 15 < q * 32) {
                    // every row of the warp lies below the chunk: exp(Acum_i - Acum_c15) gv_j,
                    // both factors <= 1
                    const float e = __expf(ai - acum[col + 15]);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        o[k] = cb[c16 * 16 + k] * e * gv[col + k];
                } else if (col > q * 32 + 31) {
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        o[k] = 0.f;
                } else {
                    // the warp's rows cross the chunk: rows below it as above; the row
                    // holding the diagonal takes exp(Acum_i - Acum_c0) hv_j when the
                    // chunk's decay span is bounded, else one exponential per element
                    const bool below = lim > 15;
                    const bool direct = !below && lim >= 0 && !sSafe[hh * 8 + (col >> 4)];
                    if (!direct) {
                        const float e = lim < 0 ? 0.f : __expf(ai - acum[below ? col + 15 : col]);
                        const float *wv = below ? gv : hv;
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            float v = k <= lim ? cb[c16 * 16 + k] * e * wv[col + k] : 0.f;
                            if (k == lim)
                                v += Dh;
                            o[k] = v;
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            float v = k <= lim ? cb[c16 * 16 + k] * __expf(ai - acum[col + k]) *
                                                     dtv[col + k]
                                               : 0.f;
                            if (k == lim)
                                v += Dh;
                            o[k] = v;
                        }
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    packed[c16 * 8 + k] = pack_bf16(o[2 * k], o[2 * k + 1]);
            }
            // bf16 pairs: K column c of the slot holds elements 2c and 2c + 1
            ptx::tmem_st8(tmem + lane_off + ls * 64 + col0 / 2, packed);
            ptx::tmem_st8(tmem + lane_off + ls * 64 + col1 / 2, packed + 8);
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(bars + kLFull + ls);
            if (mt == 0 && hh == 0)
                SSD_TRACE_EV(2, 11);
            if (mt == 64 && hh < 4)
                SSD_TRACE_EV(2, 17 + 2 * hh);
            if (mt == 0 && hh == 1)
                SSD_TRACE_EV(2, 28);
        }
        if (mt == 0)
            SSD_TRACE_EV(2, 12);

        // ---- epilogue, one off-diagonal group at a time; each 128 x 64 tile of
        //      y goes out through shared memory as whole 128-byte rows ----
        ok = !math_barrier_any(!ok);
        for (int gi = 0; gi < n_groups && ok; ++gi) {
            ok = !math_barrier_any(!ptx::mbar_wait(bars + kYoFull + gi, 0, kWaitTimeoutNs));
            if (!ok)
                break;
            ptx::tc_fence_after_sync();
            if (mt == 0 && gi == 0)
                SSD_TRACE_EV(2, 13);
            for (int hh = gi * YG; hh < group_end(gi); ++hh) {
                const float eai = has_prev ? __expf(sAcum[hh * kRows + i]) : 0.f;
                const int xoff = ((h0 + hh) * p.P - x_base) & 63;   // head's column in its X block
                const uint32_t yd_col = kColYd + hh * P_pad + xoff;
                const uint32_t yo_col = kColYo + (hh - gi * YG) * P_pad;
                __nv_bfloat16 *yh = p.y + static_cast<int64_t>(t0) * p.y_ts + (h0 + hh) * p.P;
                for (int cb0 = 0; cb0 < p.P; cb0 += 64) {
                    const int col = cb0 + quarter * 16;   // this thread's 16 columns
                    if (col < p.P) {
                        float yd[16], yo[16];
                        ptx::tmem_ld16(tmem + lane_off + yd_col + col, yd);
                        if (has_prev)
                            ptx::tmem_ld16(tmem + lane_off + yo_col + col, yo);
                        uint32_t out[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            float y0 = yd[2 * k], y1 = yd[2 * k + 1];
                            if (has_prev) {
                                y0 += eai * yo[2 * k];
                                y1 += eai * yo[2 * k + 1];
                            }
                            out[k] = pack_bf16(y0, y1);
                        }
                        uint8_t *row = sY + i * 128;
                        const int ch = quarter * 2;
                        *reinterpret_cast<uint4 *>(row + ((ch ^ (i & 7)) << 4)) =
                            make_uint4(out[0], out[1], out[2], out[3]);
                        *reinterpret_cast<uint4 *>(row + (((ch + 1) ^ (i & 7)) << 4)) =
                            make_uint4(out[4], out[5], out[6], out[7]);
                    }
                    math_barrier();
                    const int nch = (p.P - cb0 < 64 ? p.P - cb0 : 64) / 8;   // 16-byte chunks per row
                    for (int e = mt; e < kRows * 8; e += kMathThreads) {
                        const int r = e >> 3, ch = e & 7;
                        if (ch < nch && r < len) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(sY + r * 128 +
                                                                             ((ch ^ (r & 7)) << 4));
                            *reinterpret_cast<uint4 *>(yh + static_cast<int64_t>(r) * p.y_ts + cb0 +
                                                       ch * 8) = v;
                        }
                    }
                    math_barrier();
                }
            }
            // the Yoff accumulator may take the next group
            if (has_prev && gi + 1 < n_groups) {
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(bars + kYoEmpty);
            }
        }
        if (mt == 0)
            SSD_TRACE_EV(2, 14);
        if (!ok)
            *s_abort = 1;
    }

    pdl_wait();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0)
        SSD_TRACE_EV(2, 15);
    if (tid == 0 && *s_abort)
        record_error(p.hdr, kErrTimeout);
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

SmemOptIn s_smem_configured;

}  // namespace

bool use_block_table(int64_t T, int32_t batch, int H, int G, int P, int N, int Qb, int short_len)
{
    if (batch > kMapBatchMax)
        return true;
    if (batch <= 0)
        return false;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const K3Config c = chunk_scan_config(H, G, P, N);
    if (c.HB == 0)
        return false;
    // a per-CTA scan of query_start_loc costs one round trip per wave of the
    // block kernels, the block-map kernel one launch in the chain: the table
    // pays from about four waves of one CTA per SM on
    const int64_t ctas = max_chunks_bound(T, batch, Qb, short_len) * (H / c.HB);
    return ctas > 4 * static_cast<int64_t>(sms);
}

K3Config chunk_scan_config(int H, int G, int P, int N)
{
    K3Config c{};
    const int hpg = H / G;
    c.P_pad = pad64(P);
    c.N_pad = pad64(N);
    c.YG = 128 / c.P_pad;
    // heads per CTA: the largest divisor of the group's heads whose diagonal
    // accumulators fit 256 tensor-memory columns (the heads share one CB)
    const int hb_max = 256 / c.P_pad;
    for (int hb = hpg < hb_max ? hpg : hb_max; hb >= 1; --hb) {
        if (hpg % hb)
            continue;
        c.HB = hb;
        break;
    }
    // X blocks: the heads' columns from a 64-aligned start (one extra block
    // when head_dim < 64 and the start is not aligned)
    c.n_xb = (c.HB * P + 63) / 64 + (P < 64 ? 1 : 0);
    c.smem = k3_layout(c.N_pad, c.HB, c.n_xb).total + 1024;
    if (c.smem > static_cast<size_t>(kMaxSmemPerBlock))
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
    cfg.gridDim = blocks_on_y(p) ? dim3(p.H / c.HB, p.max_chunks) : dim3(p.max_chunks, p.H / c.HB);
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
