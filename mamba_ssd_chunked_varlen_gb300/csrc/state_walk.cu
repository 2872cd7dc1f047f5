// Stages 1, 2c and 3 fused for calls of long sequences with many heads: a
// persistent kernel that computes the block states and runs the inter-block
// state recurrence while walking each sequence's blocks in order, so that the
// block states never leave the chip.  The split design (chunk_state.cu, then
// state_passing.cu) writes every block state and reads it back; when those
// bytes exceed the L2 and the sequences are long enough to amortise a walk's
// start, this kernel replaces both (the host picks one per call).
//
// For every sequence b, head h and block c of b (c = 0, 1, ...):
//   dt_j      = softplus(dt[j,h] + dt_bias[h])   ("Per-token recurrence",
//   Acum_j    = A[h] (dt_0 + ... + dt_j)           Modular page "mamba2_ssd_scan";
//                                                  within the block)
//   S_c       = sum_j exp(Acum_last - Acum_j) dt_j  x_j (x) B_j   (block state)
//   S_prev[c] = S;   S = exp(Acum_last) S + S_c    (inter-chunk state recurrence)
// with S starting from the sequence's initial state (or zero) and its last
// value the final state: written into the pool slot in place (page
// "Mamba2SSDChunkScanVarlenFwdInplace") or into final_states.  These are the
// block state and the "inter-chunk state recurrence" of the chunked SSD form
// of the kernelindex page "Mamba chunk scan with segsum"; blocks are at most
// 128 tokens of one sequence, aligned to its start.
//
// A work item is (sequence, HB heads of one B group, a tile of 128 dstate
// rows).  Its CTA walks the sequence's blocks.  Per block the state is a
// dense contraction over the block's tokens on the tcgen05 tensor cores,
//   S_c^T[n, (h,p)] = sum_j Bmat[j, n] (w_j,h x[j, h, p]),
// M = 128 dstate rows, N = HB x head_dim (64 or 128 columns), K = tokens,
// into one of two tensor-memory slots; the weighted operand is formed by the
// threads in place of x, split into bf16 hi + lo (one bf16 rounding of w x
// would leave ~1e-3 relative error in final states, the split ~2^-17).  The
// running state S lives in tensor memory beside the slots, one dstate row per
// lane.  Per block only the bf16 S_prev (the chunk-scan kernel's operand) is
// written, per item the final state.
//
// Warp roles (16 warps):
//   warp 0             TMA producer: the item's B tile, x and dt of each block
//                      into a ring of stages
//   warp 1             tcgen05 issuer (owns the tensor memory)
//   warps 2, 3, 8-15   operand: processed dt, cumulative decay and weights (a
//                      warp per head), then w x as hi over x and lo beside it
//   warps 4-7          chain: S_prev out, then S = d S + S_c
// The stages run ahead of the chain by up to the ring depth; with two slots
// block c+1's MMAs overlap the chain's use of block c.
//
// Batches of at most kMapBatchMax sequences: CTA 0 does the per-call
// bookkeeping (error word, work lists for the short-sequence kernel, header)
// and every walking CTA builds the list of long sequences in shared memory
// from query_start_loc itself.  Larger batches: the block-map kernel has done
// both; the walking CTAs read its list.
#include "kernels.cuh"
#include "sm100_ptx.cuh"
#include "ssd_device.cuh"
#include "trace.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 512;
constexpr int kRows = 128;                // tokens per block tile (max)
constexpr int kBlk16 = kRows * 128;       // one 64-column x 128-row swizzled block (16 KB)
constexpr int kRowBlk = 64 * 128;         // its 64-row half (one TMA box, 8 KB)
constexpr int kOpThreads = 10 * 32;       // operand warps 2, 3, 8..15
constexpr int kChainThreads = 4 * 32;     // chain warps 4..7
constexpr int kMaxStages = 3;
constexpr int kDecRing = 8;               // per-block decays in flight (> stages + 2 + 1)
constexpr int kMaxHB = 8;                 // heads per item: HB * head_dim <= 128, head_dim >= 16

enum {
    kBarFull = 0,                         // [stage] B and x landed
    kBarOpReady = kBarFull + kMaxStages,  // [stage] weighted operand written
    kBarEmpty = kBarOpReady + kMaxStages, // [stage] its MMAs done (stage free)
    kBarScFull = kBarEmpty + kMaxStages,  // [slot] S_c final in tensor memory
    kBarScEmpty = kBarScFull + 2,         // [slot] read by the chain
    kBarDec = kBarScEmpty + 2,            // [ring] the block's decays written
    kBarDrain = kBarDec + kDecRing,       // every MMA complete (before the free)
    kNumBars = kBarDrain + 1
};

__host__ __device__ inline int walk_stages(int NP) { return NP > 64 ? 2 : 3; }

constexpr int kDtHeads = 16;              // heads of a dt box (from a multiple of 8)
constexpr int kDtRowBlk = kDtHeads * 64 * 2;   // one 64-token dt box (2 KB)

struct WalkLayout {
    uint32_t stage, sX, sL, sDt;   // a stage: B tile at 0, x (hi) at sX, lo at sL, dt at sDt
    uint32_t list, wt, dec, scratch, bars, tmem_slot, total;
};

__host__ __device__ inline WalkLayout walk_layout(int NP)
{
    WalkLayout L;
    L.sX = 2 * kBlk16;
    L.sL = L.sX + (NP / 64) * kBlk16;
    L.sDt = L.sL + (NP / 64) * kBlk16;
    L.stage = L.sDt + 2 * kDtRowBlk;
    uint32_t off = walk_stages(NP) * L.stage;
    L.list = off;
    off += kMapBatchMax * sizeof(SeqRec);
    L.wt = off;
    off += (NP / 16) * kRows * 4;   // one block's weights of up to NP / 16 heads
    L.dec = off;
    off += kDecRing * kMaxHB * 4;
    L.scratch = off;
    off += 128 * 4;
    L.bars = (off + 7) & ~7u;
    off = L.bars + kNumBars * 8;
    L.tmem_slot = off;
    off += 16;
    L.total = off;
    return L;
}

// The long sequences (more than short_len tokens) of a batch of at most
// kThreads sequences, in batch order, as records in `list`, their blocks
// numbered as map_block numbers them.  Returns (query_start_loc passed the
// checks, number of long sequences).  Called by every thread of the CTA;
// uses scratch ints 0-31.
__device__ int2 build_long_list(const ScanParams &p, SeqRec *list, int32_t *scratch)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t start = 0, len = 0, n = 0, lng = 0;
    int bad = 0;
    if (tid < p.batch) {
        start = p.qsl[tid];
        const int32_t end = p.qsl[tid + 1];
        len = end - start;
        if (len < 0 || (tid == 0 && start != 0) ||
            (tid == p.batch - 1 && static_cast<int64_t>(end) != p.T)) {
            bad = 1;
            len = 0;
        }
        lng = len > p.short_len ? 1 : 0;
        n = lng ? (len + p.Q - 1) / p.Q : 0;
    }
    const int32_t in = warp_inclusive_scan(n), il = warp_inclusive_scan(lng);
    if (lane == 31) {
        scratch[warp] = in;
        scratch[16 + warp] = il;
    }
    __syncthreads();
    int32_t bn = 0, bl = 0, tl = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const int32_t vn = scratch[w], vl = scratch[16 + w];
        bn += w < warp ? vn : 0;
        bl += w < warp ? vl : 0;
        tl += vl;
    }
    if (lng) {
        SeqRec r;
        r.t0 = start;
        r.len = len;
        r.c_begin = bn + in - n;
        r.c_end = r.c_begin + n;
        r.init = seq_init_index(p, tid);
        r.fin = seq_final_index(p, tid);
        list[bl + il - 1] = r;
    }
    bad = __syncthreads_or(bad);
    return make_int2(bad ? 0 : 1, tl);
}

// Barrier over the operand warps that also returns whether any of them passed
// true, so that they leave their loop together and none is left waiting.
__device__ __forceinline__ bool operand_barrier_any(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(kOpThreads)
        : "memory");
    return r != 0;
}

template <int kNP>
__global__ void __launch_bounds__(kThreads, 1)
    state_walk_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmDt, ScanParams p, int HB, int nT,
                      int dt_tma)
{
    constexpr int kXB = kNP / 64;            // 64-column blocks of x per stage
    constexpr uint32_t kTmemCols = kNP > 64 ? 512 : 256;  // two S_c slots and S
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const WalkLayout L = walk_layout(kNP);
    const int nst = walk_stages(kNP);
    int32_t *scratch = reinterpret_cast<int32_t *>(smem + L.scratch);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (p.table == nullptr && blockIdx.x == 0) {
        // the bookkeeping CTA
        pdl_launch_dependents();
        if (tid == 0)
            p.hdr->errors = 0u;
        const BlockInfo bi = map_block<kThreads>(p, int64_t(1) << 62, scratch, p.seq_first);
        call_bookkeeping<kThreads>(p, bi, scratch);
        return;
    }
    const int wid = blockIdx.x - (p.table == nullptr ? 1 : 0);
    const int nwalk = gridDim.x - (p.table == nullptr ? 1 : 0);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
    float *sWt = reinterpret_cast<float *>(smem + L.wt);
    float *sDec = reinterpret_cast<float *>(smem + L.dec);
    if (tid == 0)
        SSD_TRACE_EV(0, 0);

    if (tid == 0) {
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmX);
        if (dt_tma)
            ptx::prefetch_tensormap(&tmDt);
        for (int s = 0; s < nst; ++s) {
            ptx::mbar_init(bars + kBarFull + s, 1);
            ptx::mbar_init(bars + kBarOpReady + s, kOpThreads);
            ptx::mbar_init(bars + kBarEmpty + s, 1);
        }
        for (int k = 0; k < 2; ++k) {
            ptx::mbar_init(bars + kBarScFull + k, 1);
            ptx::mbar_init(bars + kBarScEmpty + k, kChainThreads);
        }
        for (int k = 0; k < kDecRing; ++k)
            ptx::mbar_init(bars + kBarDec + k, 1);
        ptx::mbar_init(bars + kBarDrain, 1);
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }

    const SeqRec *list;
    int2 vl;
    if (p.table != nullptr) {
        // the block-map kernel has listed the long sequences
        pdl_wait();
        vl = make_int2(p.hdr->valid, p.hdr->n_long);
        list = p.long_list;
    } else {
        SeqRec *s_list = reinterpret_cast<SeqRec *>(smem + L.list);
        vl = build_long_list(p, s_list, scratch);
        list = s_list;
    }
    // the chunk-scan kernel may start launching; it waits for this grid
    pdl_launch_dependents();
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int per_seq = (p.H / HB) * nT;
    const int n_items = vl.x ? vl.y * per_seq : 0;
    const int hpg = p.H / p.G;
    const int width = HB * p.P;   // valid columns of an item
    bool failed = false;
    if (tid == 0)
        SSD_TRACE_EV(0, 1);

    // item -> its sequence record, first head and dstate tile
    auto item_of = [&](int it, SeqRec &r, int &h0, int &nt) {
        r = list[it / per_seq];
        const int rem = it % per_seq;
        h0 = (rem / nT) * HB;
        nt = rem % nT;
    };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t g = 0;
            for (int it = wid; it < n_items && !failed; it += nwalk) {
                SeqRec r;
                int h0, nt;
                item_of(it, r, h0, nt);
                const int grp = h0 / hpg;
                for (int c = r.c_begin; c < r.c_end; ++c, ++g) {
                    const int s = static_cast<int>(g % nst);
                    const uint32_t use = g / nst;
                    if (use > 0 && !ptx::mbar_wait(bars + kBarEmpty + s, (use - 1) & 1, kWaitTimeoutNs)) {
                        failed = true;
                        break;
                    }
                    uint8_t *st = smem + s * L.stage;
                    const int i = c - r.c_begin;
                    const int t = r.t0 + i * p.Q;
                    const int len = min(p.Q, r.len - i * p.Q);
                    const int nrb = (len + 63) / 64;   // 64-row halves the MMAs read
                    uint64_t *full = bars + kBarFull + s;
                    ptx::mbar_arrive_expect_tx(full, nrb * ((2 + kXB) * kRowBlk + (dt_tma ? kDtRowBlk : 0)));
                    for (int rb = 0; rb < nrb; ++rb) {
                        if (dt_tma)   // dt of heads [h0 & ~7, + 16): the box starts 16-byte aligned
                            ptx::tma_load_3d(st + L.sDt + rb * kDtRowBlk, &tmDt, full, h0 & ~7,
                                             t + rb * 64, 0);
                        for (int nb = 0; nb < 2; ++nb)
                            ptx::tma_load_3d(st + nb * kBlk16 + rb * kRowBlk, &tmB, full,
                                             nt * 128 + nb * 64, grp, t + rb * 64);
                        for (int cb = 0; cb < kXB; ++cb)
                            ptx::tma_load_3d(st + L.sX + cb * kBlk16 + rb * kRowBlk, &tmX, full,
                                             h0 * p.P + cb * 64, t + rb * 64, 0);
                    }
                }
            }
            // the last loads of every stage have landed before the CTA exits
            // (they have, unless a wait above gave up)
            for (int s = 0; s < nst; ++s)
                if (g > static_cast<uint32_t>(s)) {
                    const uint32_t last = (g - 1 - s) / nst;
                    if (!ptx::mbar_wait(bars + kBarFull + s, last & 1, kWaitTimeoutNs))
                        failed = true;
                }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(128, kNP, 1, 1);
            uint32_t g = 0;
            for (int it = wid; it < n_items && !failed; it += nwalk) {
                SeqRec r;
                int h0, nt;
                item_of(it, r, h0, nt);
                for (int c = r.c_begin; c < r.c_end; ++c, ++g) {
                    const int s = static_cast<int>(g % nst);
                    const uint32_t use = g / nst;
                    const int slot = static_cast<int>(g & 1);
                    const uint32_t suse = g >> 1;
                    if (!ptx::mbar_wait(bars + kBarOpReady + s, use & 1, kWaitTimeoutNs) ||
                        (suse > 0 &&
                         !ptx::mbar_wait(bars + kBarScEmpty + slot, (suse - 1) & 1, kWaitTimeoutNs))) {
                        failed = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const int i = c - r.c_begin;
                    const int len = min(p.Q, r.len - i * p.Q);
                    const uint32_t sb = ptx::smem_u32(smem + s * L.stage);
                    const uint64_t dA = ptx::sdesc_sw128(sb, kBlk16, 1024);
                    const uint64_t dH = ptx::sdesc_sw128(sb + L.sX, kBlk16, 1024);
                    const uint64_t dL = ptx::sdesc_sw128(sb + L.sL, kBlk16, 1024);
                    const uint32_t d = tmem + slot * kNP;
                    const int nks = (len + 15) / 16;
                    for (int ks = 0; ks < nks; ++ks) {
                        const uint32_t o = ks * 2048;   // 16 token rows
                        ptx::mma_bf16_ss(d, ptx::sdesc_add(dA, o), ptx::sdesc_add(dH, o), idesc, ks > 0);
                        ptx::mma_bf16_ss(d, ptx::sdesc_add(dA, o), ptx::sdesc_add(dL, o), idesc, 1);
                    }
                    ptx::mma_commit(bars + kBarEmpty + s);
                    ptx::mma_commit(bars + kBarScFull + slot);
                }
            }
            if (g > 0) {
                ptx::mma_commit(bars + kBarDrain);
                if (!ptx::mbar_wait(bars + kBarDrain, 0, kWaitTimeoutNs))
                    failed = true;
            }
        }
    } else if (warp < 4 || warp >= 8) {
        // ---------------------------------------------------------- operand
        const int ow = warp < 4 ? warp - 2 : warp - 6;   // 0..9
        const int ot = ow * 32 + lane;
        const int log2P = __ffs(p.P) - 1;
        uint32_t g = 0;
        for (int it = wid; it < n_items && !failed; it += nwalk) {
            SeqRec r;
            int h0, nt;
            item_of(it, r, h0, nt);
            // warp ow computes the weights of head ow of the item
            const bool scan_warp = ow < HB;
            const float Ah = scan_warp ? p.A[h0 + ow] : 0.f;
            const float bias = (scan_warp && p.dt_bias) ? p.dt_bias[h0 + ow] : 0.f;
            for (int c = r.c_begin; c < r.c_end; ++c, ++g) {
                const int s = static_cast<int>(g % nst);
                const uint32_t use = g / nst;
                const int i = c - r.c_begin;
                const int64_t t = r.t0 + static_cast<int64_t>(i) * p.Q;
                const int len = min(p.Q, r.len - i * p.Q);
                uint8_t *st = smem + s * L.stage;
                float *dec = sDec + (g % kDecRing) * kMaxHB;
                // the stage's tiles (and dt); the decision to go on is the same for
                // every operand warp (this barrier also ends the previous block's
                // reads of the weights)
                const bool ok = ptx::mbar_wait(bars + kBarFull + s, use & 1, kWaitTimeoutNs);
                if (operand_barrier_any(!ok)) {
                    failed = true;
                    break;
                }
                // dt, cumulative A dt and the weights exp(Acum_last - Acum_j) dt_j:
                // one warp per head, four tokens per lane
                if (scan_warp) {
                    const __nv_bfloat16 *sdt =
                        reinterpret_cast<const __nv_bfloat16 *>(st + L.sDt) + (h0 & 7) + ow;
                    float dv[4], acc[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 4 * lane + e;
                        float v = 0.f;
                        if (j < len) {
                            v = __bfloat162float(dt_tma ? sdt[j * kDtHeads]
                                                        : p.dt[(t + j) * p.dt_ts + h0 + ow]) + bias;
                            v = p.dt_softplus ? softplus_f32(v) : v;
                        }
                        dv[e] = v;
                    }
                    float run = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        run += Ah * dv[e];
                        acc[e] = run;
                    }
                    const float excl = warp_inclusive_scan(run) - run;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc[e] += excl;
                    const int le = (len - 1) & 3;
                    const float mine = le == 0 ? acc[0] : le == 1 ? acc[1] : le == 2 ? acc[2] : acc[3];
                    const float last = __shfl_sync(0xffffffffu, mine, (len - 1) >> 2);
                    float4 w4;
                    w4.x = 4 * lane + 0 < len ? expf(last - acc[0]) * dv[0] : 0.f;
                    w4.y = 4 * lane + 1 < len ? expf(last - acc[1]) * dv[1] : 0.f;
                    w4.z = 4 * lane + 2 < len ? expf(last - acc[2]) * dv[2] : 0.f;
                    w4.w = 4 * lane + 3 < len ? expf(last - acc[3]) * dv[3] : 0.f;
                    reinterpret_cast<float4 *>(sWt + ow * kRows)[lane] = w4;
                    if (lane == 0)
                        dec[ow] = expf(last);
                }
                operand_barrier_any(false);   // every head's weights and decay written
                if (ot == 0)
                    ptx::mbar_arrive(bars + kBarDec + g % kDecRing);
                // the weighted operand, hi over x in place and lo beside it, for the
                // rows the MMAs read (zero past the block end and past the heads);
                // two 16-byte chunks per thread in flight
                uint8_t *sx = st + L.sX;
                uint8_t *sl = st + L.sL;
                const int nrows = (len + 15) & ~15;
                constexpr int kChunks = kNP / 8;   // 16-byte chunks per row
                const int n_idx = nrows * kChunks;
                auto chunk_off = [&](int idx, int &row, int &c0) -> uint32_t {
                    row = idx / kChunks;
                    c0 = (idx % kChunks) * 8;
                    return (c0 >> 6) * kBlk16 + (row >> 3) * 1024 + (row & 7) * 128 +
                           ((((c0 & 63) >> 3) ^ (row & 7)) << 4);
                };
                auto hilo = [&](const uint4 &raw, int row, int c0, uint4 &hi4, uint4 &lo4) {
                    uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
                    if (row < len && c0 < width) {
                        const __nv_bfloat162 *xb = reinterpret_cast<const __nv_bfloat162 *>(&raw);
                        const float w = sWt[(c0 >> log2P) * kRows + row];
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
                for (int idx = ot; idx < n_idx; idx += 2 * kOpThreads) {
                    const int idx2 = idx + kOpThreads;
                    int r0, c00, r1 = 0, c01 = 0;
                    const uint32_t o0 = chunk_off(idx, r0, c00);
                    const uint32_t o1 = idx2 < n_idx ? chunk_off(idx2, r1, c01) : 0u;
                    const uint4 raw0 = *reinterpret_cast<const uint4 *>(sx + o0);
                    uint4 raw1 = make_uint4(0u, 0u, 0u, 0u);
                    if (idx2 < n_idx)
                        raw1 = *reinterpret_cast<const uint4 *>(sx + o1);
                    uint4 hi4, lo4;
                    hilo(raw0, r0, c00, hi4, lo4);
                    *reinterpret_cast<uint4 *>(sx + o0) = hi4;
                    *reinterpret_cast<uint4 *>(sl + o0) = lo4;
                    if (idx2 < n_idx) {
                        hilo(raw1, r1, c01, hi4, lo4);
                        *reinterpret_cast<uint4 *>(sx + o1) = hi4;
                        *reinterpret_cast<uint4 *>(sl + o1) = lo4;
                    }
                }
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(bars + kBarOpReady + s);
            }
        }
    } else {
        // ---------------------------------------------------------- chain
        // warps 4..7: tensor-memory lane quarter q holds dstate rows q*32 ..;
        // the running state S lives in tensor memory beside the two S_c slots
        const int q = warp & 3;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t s_col = 2 * kNP;
        const int log2P = __ffs(p.P) - 1;
        const int64_t PN = static_cast<int64_t>(p.P) * p.N;
        uint32_t g = 0;
        for (int it = wid; it < n_items && !failed; it += nwalk) {
            SeqRec r;
            int h0, nt;
            item_of(it, r, h0, nt);
            const int n = nt * 128 + q * 32 + lane;
            const bool nv = n < p.N;
            // column c = hh P + p of the item is element (h0 P + c) N + n of a
            // [head][p][n] state (pool slot or entering state)
            const int64_t e0 = static_cast<int64_t>(h0) * PN + n;
            // the initial state (or zero) into tensor memory, 16 columns at a time
            for (int c16 = 0; c16 < kNP; c16 += 16) {
                uint32_t v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int col = c16 + k;
                    float f = 0.f;
                    if (r.init >= 0 && nv && col < width)
                        f = load_init1(p, r.init + e0 + static_cast<int64_t>(col) * p.N);
                    v[k] = __float_as_uint(f);
                }
                ptx::tmem_st16(lane_base + s_col + c16, v);
            }
            ptx::tmem_wait_st();
            for (int blk = r.c_begin; blk < r.c_end; ++blk, ++g) {
                const int slot = static_cast<int>(g & 1);
                if (!ptx::mbar_wait_sleep(bars + kBarScFull + slot, (g >> 1) & 1, kWaitTimeoutNs, 64) ||
                    !ptx::mbar_wait_sleep(bars + kBarDec + g % kDecRing, (g / kDecRing) & 1,
                                          kWaitTimeoutNs, 64)) {
                    failed = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                const float *dec = sDec + (g % kDecRing) * kMaxHB;
                const bool last = blk == r.c_end - 1;
                // the state entering the block goes out as the chunk-scan kernel's
                // bf16 operand (a first block without initial state is taken as
                // zero there); then S = d S + S_c, or the final state after the
                // last block
                const bool put_prev = nv && (blk != r.c_begin || r.init >= 0);
                __nv_bfloat16 *sp = p.sprev + static_cast<int64_t>(blk) * p.H * PN + e0;
                for (int c16 = 0; c16 < kNP && c16 < width; c16 += 16) {
                    float sc[16], sv[16];
                    ptx::tmem_ld16(lane_base + slot * kNP + c16, sc);
                    ptx::tmem_ld16(lane_base + s_col + c16, sv);
                    // 16 columns never straddle two heads (head_dim >= 16)
                    const float d = dec[c16 >> log2P];
                    if (put_prev) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            sp[static_cast<int64_t>(c16 + k) * p.N] = __float2bfloat16_rn(sv[k]);
                    }
                    uint32_t nv16[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        nv16[k] = __float_as_uint(fmaf(d, sv[k], sc[k]));
                    if (!last) {
                        ptx::tmem_st16(lane_base + s_col + c16, nv16);
                    } else if (r.fin >= 0 && nv) {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            store_final1(p, r.fin + e0 + static_cast<int64_t>(c16 + k) * p.N,
                                         __uint_as_float(nv16[k]));
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before_sync();
                ptx::mbar_arrive(bars + kBarScEmpty + slot);
            }
        }
    }

    if (failed)
        record_error(p.hdr, kErrTimeout);
    if (tid == 0)
        SSD_TRACE_EV(0, 2);
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

SmemOptIn s_smem_64, s_smem_128;

}  // namespace

bool use_state_walk(int64_t T, int32_t batch, int H, int G, int P, int N, int Qb)
{
    if (batch <= 0 || T < static_cast<int64_t>(2048) * batch)
        return false;
    int dev = 0, sms = 152, l2 = 126 << 20;
    if (cudaGetDevice(&dev) == cudaSuccess) {
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    }
    const WalkConfig c = state_walk_config(H, G, P, N, batch, sms);
    if (static_cast<int64_t>(batch) * (H / c.HB) * c.nT < sms)
        return false;
    // the split design's block states (fp16) and entering states (bf16): 4 bytes
    // per state element and block
    const int64_t state_bytes = (T + Qb - 1) / Qb * static_cast<int64_t>(H) * P * N * 4;
    return state_bytes > l2;
}

WalkConfig state_walk_config(int H, int G, int P, int N, int batch, int sms)
{
    WalkConfig c{};
    const int hpg = H / G;
    c.nT = (N + 127) / 128;
    // heads per item: the most whose columns fit one 128-column slot while the
    // batch still gives every SM an item; one head when it gives fewer
    c.HB = 1;
    for (int hb = 2; hb <= hpg && hb <= kMaxHB && hb * P <= 128; ++hb) {
        if (hpg % hb)
            continue;
        if (static_cast<int64_t>(batch) * (H / hb) * c.nT >= sms)
            c.HB = hb;
    }
    c.NP = pad64(c.HB * P);
    c.smem = walk_layout(c.NP).total + 1024;
    return c;
}

cudaError_t launch_state_walk(const ScanParams &p, const StateWalkMaps &maps, cudaStream_t stream,
                              bool programmatic)
{
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const WalkConfig c = state_walk_config(p.H, p.G, p.P, p.N, p.batch, sms);
    const void *kernel = c.NP > 64 ? reinterpret_cast<const void *>(state_walk_kernel<128>)
                                   : reinterpret_cast<const void *>(state_walk_kernel<64>);
    cudaError_t e = ensure_max_smem(kernel, c.NP > 64 ? s_smem_128 : s_smem_64);
    if (e != cudaSuccess)
        return e;
    // one walking CTA per item up to one per SM (each loops over items beyond
    // that), plus the bookkeeping CTA when there is no block-map kernel
    const int64_t items = static_cast<int64_t>(p.batch) * (p.H / c.HB) * c.nT;
    const int64_t walkers = items < sms ? items : sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(walkers + (p.table == nullptr ? 1 : 0)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (c.NP > 64)
        return cudaLaunchKernelEx(&cfg, state_walk_kernel<128>, maps.B, maps.X, maps.Dt, p, c.HB,
                                  c.nT, maps.dt_tma);
    return cudaLaunchKernelEx(&cfg, state_walk_kernel<64>, maps.B, maps.X, maps.Dt, p, c.HB, c.nT,
                              maps.dt_tma);
}

}  // namespace ssd
