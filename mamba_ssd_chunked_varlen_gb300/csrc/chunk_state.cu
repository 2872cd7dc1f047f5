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
// x arrive by TMA (MN-major, 128-byte swizzle); B is used as it is, shared by
// the heads.  The weighted operand w_j x_j is formed by the threads in place
// of x and split into bf16 hi + lo parts (two MMAs into one fp32 accumulator):
// one bf16 rounding of w x would leave ~1e-3 relative error in final states,
// the split leaves ~2^-17.  The CTA maps its block to its sequence itself, and
// CTA (0,0) writes the per-sequence first-block table and resets the error word.
//
// Block states are stored [block][head][p][n] like the pool's slots, so the
// state-passing kernel reads and writes both with the same coalesced pattern;
// they cross the workspace as fp16 with a power-of-two exponent per 16
// consecutive p (state_group_exp), half the bytes of fp32.
#include "kernels.cuh"
#include "sm100_ptx.cuh"
#include "ssd_device.cuh"
#include "trace.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 512;
constexpr int kRows = 128;                     // tokens per block (max)
constexpr int kNBlockBytes = kRows * 128;      // one 64-wide block of 128 rows (16 KB)

struct K1Layout {
    uint32_t sB, sW, sLo, sDt, sAcum, sWt, scratch, bars, tmem_slot, total;
};

__host__ __device__ inline K1Layout k1_layout(int NP, int n_mtiles, int HB)
{
    K1Layout L;
    uint32_t off = 0;
    L.sB = off;
    off += n_mtiles * 2 * kNBlockBytes;
    L.sW = off;
    off += (NP / 64) * kNBlockBytes;
    L.sLo = off;
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
    off = L.bars + 5 * 8;
    L.tmem_slot = off;
    off += 16;
    L.total = off;
    return L;
}

// Batches of more than kMapBatchMax sequences: one CTA maps every block once
// into the block table (and does the bookkeeping); the block kernels, launched
// as its programmatic dependents, look their block up instead of scanning
// query_start_loc each.
__global__ void __launch_bounds__(kThreads) block_map_kernel(ScanParams p)
{
    __shared__ int32_t scratch[64];
    // the chunk-state kernel may start launching; it waits for this grid
    pdl_launch_dependents();
    if (threadIdx.x == 0)
        p.hdr->errors = 0u;
    // a block index past every block: the scan only writes the tables
    const BlockInfo bi = map_block<kThreads>(p, int64_t(1) << 62, scratch, p.seq_first, p.table);
    call_bookkeeping<kThreads>(p, bi, scratch);
}

// kFinishSingle: a sequence's only block is finished here (batches of several
// sequences); without it every block state goes to the state-passing kernel
// and the kernel keeps to 64 registers, so that two state-passing CTAs wait
// beside it.
template <bool kFinishSingle>
__global__ void __launch_bounds__(kThreads, kFinishSingle ? 1 : 2)
    chunk_state_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmX,
                       ScanParams p, int HB, int NP, int n_mtiles, uint32_t tmem_cols)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const K1Layout L = k1_layout(NP, n_mtiles, HB);
    uint8_t *sB = smem + L.sB;
    uint8_t *sW = smem + L.sW;
    uint8_t *sLo = smem + L.sLo;
    float *sDt = reinterpret_cast<float *>(smem + L.sDt);
    float *sAcum = reinterpret_cast<float *>(smem + L.sAcum);
    float *sWt = reinterpret_cast<float *>(smem + L.sWt);
    int32_t *scratch = reinterpret_cast<int32_t *>(smem + L.scratch);
    uint64_t *bar_b = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *bar_x = bar_b + 1;
    uint64_t *bar_mma = bar_b + 2;   // one per state tile (n_mtiles <= 2)
    uint64_t *bar_never = bar_b + 4;  // completed by nothing (the bounded-wait test)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
    float *s_part = reinterpret_cast<float *>(scratch + 40);  // 16 warp partials

    const bool by_rows = blocks_on_y(p);
    const int blk = by_rows ? blockIdx.y : blockIdx.x;
    const int h0 = (by_rows ? blockIdx.x : blockIdx.y) * HB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The per-call bookkeeping (block table, error word, slot checks) falls to
    // CTA (max_chunks - 1, 0): max_chunks bounds the number of blocks from
    // above with its last index always free, so that CTA never holds a block
    // and the bookkeeping delays no block's work.
    const bool leader = blockIdx.x == gridDim.x - 1 && blockIdx.y == 0;
    if (tid == 0)
        SSD_TRACE_EV(0, 0);

    if (tid == 0) {
        // descriptors fetched while the block is being mapped
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmX);
    }
    BlockInfo bi;
    if (p.table != nullptr) {
        // the block-map kernel has mapped every block (and done the bookkeeping)
        pdl_wait();
        bi = lookup_block(p, blk);
    } else {
        if (leader && tid == 0)
            p.hdr->errors = 0u;
        bi = map_block<kThreads>(p, blk, scratch, leader ? p.seq_first : nullptr);
        if (leader)
            call_bookkeeping<kThreads>(p, bi, scratch);
    }
    // the state-passing kernel may start launching; it waits for this grid
    // (with the block table, only once this CTA has read it, so that every
    // later kernel finds the block-map kernel complete)
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
        ptx::mbar_init(bar_never, 1);
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
    //      once (one round trip), then four heads per scan pass ----
    const int quarter = tid >> 7, j = tid & 127;
    float dv[2], av[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int hh = 4 * k + quarter;
        dv[k] = (hh < HB && j < len) ? processed_dt(p, t0 + j, h0 + hh) : 0.f;
        av[k] = hh < HB ? p.A[h0 + hh] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if (4 * k >= HB)
            break;
        const int hh = 4 * k + quarter;
        const float incl = warp_inclusive_scan(av[k] * dv[k]);
        if (lane == 31)
            s_part[warp] = incl;
        __syncthreads();
        float before = 0.f;
        for (int w = quarter * 4; w < warp; ++w)
            before += s_part[w];
        if (hh < HB) {
            sDt[hh * kRows + j] = dv[k];
            sAcum[hh * kRows + j] = before + incl;
        }
        __syncthreads();
    }
    for (int i = tid; i < HB * kRows; i += kThreads) {
        const int hh = i / kRows, jj = i % kRows;
        const float last = sAcum[hh * kRows + len - 1];
        const float w = jj < len ? expf(last - sAcum[i]) * sDt[i] : 0.f;
        sWt[i] = w;
        if (jj == 0)
            p.decay[static_cast<int64_t>(blk) * p.H + h0 + hh] = expf(last);
    }
    if (tid == 0)
        SSD_TRACE_EV(0, 2);

    bool failed = !(ptx::mbar_wait(bar_x, 0, kWaitTimeoutNs) && ptx::mbar_wait(bar_b, 0, kWaitTimeoutNs));
    // the tests of the bounded-wait path: once the loads have landed (no copy
    // is in flight), one thread waits for a barrier that nothing completes;
    // the wait gives up after test_stall_ns and the CTA takes the timeout path
    if (p.test_stall_ns != 0 && tid == 0 && !failed)
        failed = !ptx::mbar_wait(bar_never, 0, p.test_stall_ns);
    failed = __syncthreads_or(failed);
    if (tid == 0)
        SSD_TRACE_EV(0, 3);

    const int chunks8 = NP / 8;            // 16-byte chunks per token row of x
    const int width = HB * p.P;            // valid columns
    const int log2P = __ffs(p.P) - 1;
    // weighted input w_j x_j of one 16-byte chunk (8 columns) of row r, split
    // into bf16 hi + lo; zero past the block end and past the CTA's heads
    auto hilo = [&](const uint4 &raw, int r, int c0, uint4 &hi4, uint4 &lo4) {
        uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
        if (r < len && c0 < width) {
            const __nv_bfloat162 *xb = reinterpret_cast<const __nv_bfloat162 *>(&raw);
            const float w = sWt[(c0 >> log2P) * kRows + r];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 xf = __bfloat1622float2(xb[k]);
                const float v0 = w * xf.x, v1 = w * xf.y;
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(v0, v1);
                const float2 hf = __bfloat1622float2(h2);
                const __nv_bfloat162 l2 = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
                hi[k] = *reinterpret_cast<const uint32_t *>(&h2);
                lo[k] = *reinterpret_cast<const uint32_t *>(&l2);
            }
        }
        hi4 = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        lo4 = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    };
    auto swz = [&](int r, int c0) -> uint32_t {
        return (c0 >> 6) * kNBlockBytes + (r >> 3) * 1024 + (r & 7) * 128 +
               ((((c0 & 63) >> 3) ^ (r & 7)) << 4);
    };
    if (!failed) {
        // ---- the weighted operand, hi over x in place, lo beside it ----
        if ((chunks8 & (chunks8 - 1)) == 0) {
            // each thread keeps one column chunk and takes rows r0, r0 + rstep, ...;
            // four rows are loaded before any of them is rewritten
            const int lc = __ffs(chunks8) - 1;
            const int c0 = (tid & (chunks8 - 1)) * 8;
            const int rstep = kThreads >> lc;
#pragma unroll 1
            for (int r0 = tid >> lc; r0 < kRows; r0 += 4 * rstep) {
                uint4 raw[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (r0 + k * rstep < kRows)
                        raw[k] = *reinterpret_cast<const uint4 *>(sW + swz(r0 + k * rstep, c0));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (r0 + k * rstep < kRows) {
                        const int r = r0 + k * rstep;
                        uint4 hi4, lo4;
                        hilo(raw[k], r, c0, hi4, lo4);
                        *reinterpret_cast<uint4 *>(sW + swz(r, c0)) = hi4;
                        *reinterpret_cast<uint4 *>(sLo + swz(r, c0)) = lo4;
                    }
            }
        } else {
            for (int item = tid; item < kRows * chunks8; item += kThreads) {
                const int r = item / chunks8, c0 = (item % chunks8) * 8;
                const uint4 raw = *reinterpret_cast<const uint4 *>(sW + swz(r, c0));
                uint4 hi4, lo4;
                hilo(raw, r, c0, hi4, lo4);
                *reinterpret_cast<uint4 *>(sW + swz(r, c0)) = hi4;
                *reinterpret_cast<uint4 *>(sLo + swz(r, c0)) = lo4;
            }
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
        const uint32_t idesc = ptx::idesc_bf16_f32(128, NP, 1, 1);
        const uint64_t dB0 = ptx::sdesc_sw128(ptx::smem_u32(sB), kNBlockBytes, 1024);
        const uint64_t dH0 = ptx::sdesc_sw128(ptx::smem_u32(sW), kNBlockBytes, 1024);
        const uint64_t dL0 = ptx::sdesc_sw128(ptx::smem_u32(sLo), kNBlockBytes, 1024);
        const int nks = (len + 15) / 16;
        for (int mt = 0; mt < n_mtiles; ++mt) {
            const uint32_t d = tmem + mt * NP;
            const uint64_t dBm = ptx::sdesc_add(dB0, mt * 2 * kNBlockBytes);
            ptx::mma_bf16_ss(d, dBm, dH0, idesc, 0);
            ptx::mma_bf16_ss(d, dBm, dL0, idesc, 1);
            for (int ks = 1; ks < nks; ++ks) {
                const uint64_t dBk = ptx::sdesc_add(dBm, ks * 2048);
                ptx::mma_bf16_ss(d, dBk, ptx::sdesc_add(dH0, ks * 2048), idesc, 1);
                ptx::mma_bf16_ss(d, dBk, ptx::sdesc_add(dL0, ks * 2048), idesc, 1);
            }
            // each state tile is stored as soon as its accumulator is final
            ptx::mma_commit(bar_mma + mt);
        }
    }

    if (!failed) {
        // ---- epilogue: S^T tile [n][(h,p)] -> S_c[blk][h][p][n] ----
        // A sequence's only block is finished here instead of in the state-
        // passing kernel, with the same arithmetic: the entering state is the
        // initial state (its bf16 copy goes to S_prev for the chunk-scan
        // kernel), the final state decay * initial + S_c goes to its slot.
        // The initial state is loaded before the MMAs are waited for.
        const bool single = kFinishSingle && bi.first && bi.last;
        const int64_t init_i = single ? seq_init_index(p, bi.seq) : -1;
        const int64_t fin_i = single ? seq_final_index(p, bi.seq) : -1;
        const int q = warp & 3, cq = warp >> 2;  // TMEM lane quarter, column quarter
        const int ncols = NP / 4;                // <= 64: at most 4 chunks of 16
        for (int mt = 0; mt < n_mtiles && !failed; ++mt) {
            const int n = mt * 128 + q * 32 + lane;
            if (!single) {
                if (!ptx::mbar_wait(bar_mma + mt, 0, kWaitTimeoutNs)) {
                    failed = true;
                    break;
                }
                ptx::tc_fence_after_sync();
#pragma unroll 1
                for (int c = cq * ncols; c < (cq + 1) * ncols; c += 16) {
                    float v[16];
                    ptx::tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + mt * NP + c, v);
                    if (n < p.N && c < width) {
                        // 16 columns never straddle two heads (head_dim % 16 == 0) and
                        // start on a multiple of 16 of p: one exponent group.  A warp
                        // writes 32 consecutive n of one p: 64 contiguous bytes
                        const int hh = c / p.P, p0 = c % p.P;
                        const int64_t hrow = static_cast<int64_t>(blk) * p.H + h0 + hh;
                        __half *dst = p.schunk + (hrow * p.P + p0) * p.N + n;
                        float m = 0.f;
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            m = fmaxf(m, fabsf(v[k]));
                        const int ke = state_group_exp(m);
                        const float sc = pow2i(ke);
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            dst[static_cast<int64_t>(k) * p.N] = __float2half_rn(v[k] * sc);
                        p.sexp[(hrow * (p.P / 16) + p0 / 16) * p.N + n] = static_cast<int8_t>(ke);
                    }
                }
                continue;
            }
            if constexpr (kFinishSingle) {
                // the initial state of all this thread's columns is loaded
                // before the MMAs are waited for
                float iv[4][16];
                if (init_i >= 0) {
#pragma unroll
                    for (int ci = 0; ci < 4; ++ci) {
                        const int c = cq * ncols + ci * 16;
                        if (ci * 16 < ncols && n < p.N && c < width) {
                            const int64_t e =
                                (static_cast<int64_t>(h0 + c / p.P) * p.P + c % p.P) * p.N + n;
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                iv[ci][k] = load_init1(p, init_i + e + static_cast<int64_t>(k) * p.N);
                        }
                    }
                }
                if (!ptx::mbar_wait(bar_mma + mt, 0, kWaitTimeoutNs)) {
                    failed = true;
                    break;
                }
                ptx::tc_fence_after_sync();
#pragma unroll
                for (int ci = 0; ci < 4; ++ci) {
                    if (ci * 16 >= ncols)
                        break;
                    const int c = cq * ncols + ci * 16;
                    float v[16];
                    ptx::tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + mt * NP + c, v);
                    // the block state rounded as it crosses the workspace for a longer
                    // sequence (fp16 with the group's exponent), so that a sequence
                    // finished here and one continued from its slot see the same values
                    round_state_group(v);
                    if (n < p.N && c < width) {
                        const int hh = c / p.P, p0 = c % p.P;
                        const int64_t row = (static_cast<int64_t>(blk) * p.H + h0 + hh) * p.P + p0;
                        const float d = expf(sAcum[hh * kRows + len - 1]);
                        const int64_t e = (static_cast<int64_t>(h0 + hh) * p.P + p0) * p.N + n;
                        __nv_bfloat16 *sp = p.sprev + row * p.N + n;
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const float s0 = init_i >= 0 ? iv[ci][k] : 0.f;
                            if (init_i >= 0)
                                sp[static_cast<int64_t>(k) * p.N] = __float2bfloat16_rn(s0);
                            if (fin_i >= 0)
                                store_final1(p, fin_i + e + static_cast<int64_t>(k) * p.N,
                                             fmaf(d, s0, v[k]));
                        }
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

SmemOptIn s_smem_configured, s_smem_configured_single;

}  // namespace

K1Config chunk_state_config(int H, int G, int P, int N)
{
    K1Config c{};
    const int hpg = H / G;
    c.n_mtiles = (N + 127) / 128;
    // heads per CTA: as many as one MMA's columns hold (<= 256; the tensor
    // core is most efficient at N = 256 and B is shared), at most 8 heads
    // (the dt prologue holds 2 per thread)
    for (int hb = hpg < 8 ? hpg : 8; hb >= 1; --hb) {
        if (hpg % hb)
            continue;
        const int np = pad64(hb * P);
        if ((np > 256 || c.n_mtiles * np > 512) && hb > 1)
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

cudaError_t launch_block_map(const ScanParams &p, cudaStream_t stream)
{
    block_map_kernel<<<1, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_chunk_state(const ScanParams &p, const ChunkStateMaps &maps,
                               cudaStream_t stream, bool programmatic)
{
    const K1Config c = chunk_state_config(p.H, p.G, p.P, p.N);
    const void *kernel = p.finish_single
                             ? reinterpret_cast<const void *>(chunk_state_kernel<true>)
                             : reinterpret_cast<const void *>(chunk_state_kernel<false>);
    cudaError_t e = ensure_max_smem(kernel, p.finish_single ? s_smem_configured_single
                                                            : s_smem_configured);
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
    if (p.finish_single)
        return cudaLaunchKernelEx(&cfg, chunk_state_kernel<true>, maps.B, maps.X, p, c.HB, c.NP,
                                  c.n_mtiles, c.tmem_cols);
    return cudaLaunchKernelEx(&cfg, chunk_state_kernel<false>, maps.B, maps.X, p, c.HB, c.NP,
                              c.n_mtiles, c.tmem_cols);
}

}  // namespace ssd
