// Short sequences (at most p.short_len = 12 tokens): the whole scan by the
// "Per-token recurrence" of the Modular page "mamba2_ssd_scan", token by
// token, for every (sequence, head):
//
//   dt_t = softplus(dt + dt_bias);   dA_t = exp(A[h] dt_t)
//   S    = S dA_t + dt_t x_t (x) B_t          S from the initial state (or 0)
//   y_t  = C_t . S + D[h] x_t
//   final state <- S
//
// A short sequence's cost is its state: the slot read (with an initial state)
// and written, head_dim x dstate values per head, against a few tokens of x,
// B, C and y (serving batches, where most sequences are a few tokens long,
// are bound by exactly this read-modify-write: the decode note of the page
// "Mamba2SSDChunkScanVarlenFwdInplace").  So the kernel is a copy pipeline:
//
// * work items are tiles of R head_dim rows (R x dstate <= 4096 elements) of
//   one (short sequence, head); a persistent grid, one CTA per SM, gives each
//   CTA a contiguous range of items (so consecutive items share a sequence);
// * a loader warp streams each item's state tile (one bulk copy) and its
//   tokens' B, C and x rows (tensor copies of 8-token boxes) into one of the
//   shared-memory stages (mbarrier completion; as many stages as fit, sized
//   for the dstate), with the item's processed dt values copied from a table
//   it builds once per sequence (and per 128 heads);
// * two groups of 8 consumer warps take alternate items, so that one item's
//   dependent chain (loads, updates, reductions, stores) overlaps the
//   other's; on its item each thread holds a block of RB head_dim rows x NB
//   dstate values (4 x 4, or 2 x 8 at dstate > 128), so every B, C and x
//   value it unpacks serves several state elements; the RB row sums of C.S
//   of 4 tokens at a time are reduced over the row group's lanes in one
//   butterfly (each step halves the values a lane holds); y is stored
//   directly;
// * a storer warp writes each finished tile back to its slot with a bulk store
//   and frees a stage once its store has read it, with kStoreLag stores in
//   flight so that it never waits on the one it just issued.
//
// The sequences come from the list the per-call bookkeeping CTA wrote (in the
// chunk-state kernel, the fused walk or the block-map kernel; one 32-byte
// record each); the chunked kernels give them no block.
#include "kernels.cuh"
#include "sm100_ptx.cuh"
#include "ssd_device.cuh"

namespace ssd {
namespace {

constexpr int kGroupWarps = 8;              // consumer warps on one item
constexpr int kConsumerGroups = 2;          // items in work at once, alternating
constexpr int kConsumerWarps = kGroupWarps * kConsumerGroups;
constexpr int kConsumers = kGroupWarps * 32;   // threads on one item
constexpr int kThreads = kConsumerWarps * 32 + 64;   // + the loader and the storer warp
constexpr int kLoaderWarp = kConsumerWarps, kStorerWarp = kConsumerWarps + 1;
constexpr int kMaxStages = 8;
constexpr int kTabHeads = 128;              // heads per processed-dt table
constexpr int kBox = 8;                     // tokens per tensor copy
constexpr int kTokRows = (kShortLenMax + kBox - 1) / kBox * kBox;   // token rows per stage
constexpr int kTileElems = 4096;            // state elements per tile (16 KB in fp32)
constexpr int kElemsPerThread = 16;         // RB x NB
constexpr int kStoreLag = 2;                // bulk stores in flight before a stage is freed
constexpr int kGroup = 4;                   // tokens whose row sums are reduced together
constexpr size_t kSmemBytes = 225 * 1024;   // dynamic shared memory of the CTA

struct alignas(16) StageMeta {
    int32_t t0, len, h, row0;
    int32_t has_init;
    float Dh;
    int64_t fin;   // element index of the tile in the final-state storage (-1: none)
};

// The fixed part of shared memory: barriers, the error flag, the loader's
// table of processed dt and exp(A dt) per (token, head) and D per head.
constexpr int kOffBars = 0;   // full, done, empty: kMaxStages each
constexpr int kOffFailed = kOffBars + 3 * kMaxStages * 8;
constexpr int kOffTab = kOffFailed + 16;
constexpr int kOffTabD = kOffTab + kTokRows * kTabHeads * 8;
constexpr int kOffStages = (kOffTabD + kTabHeads * 4 + 127) / 128 * 128;

// Rows per tile: the largest power of two that divides head_dim (itself a
// power of two) with rows x dstate <= kTileElems.  With the dstate lanes of a
// row padded to a power of two, rows x padded dstate <= 4096, so the tile
// takes at most kConsumers threads of kElemsPerThread elements.
__host__ __device__ inline int tile_rows(int P, int N)
{
    int r = 1;
    while (2 * r <= P && 2 * r * N <= kTileElems)
        r *= 2;
    return r;
}

__host__ __device__ inline int pow2_at_least(int v)
{
    int r = 1;
    while (r < v)
        r *= 2;
    return r;
}

// One pipeline stage, sized for the call's tile and dstate: the state tile,
// the tokens' B, C (bf16 [token][N]) and x rows (bf16 [token][R]), the
// processed dt and exp(A dt) per token, the item's description.
struct StageLayout {
    int offB, offC, offX, offDt, offMeta, bytes, count;
};

__host__ __device__ inline StageLayout stage_layout(int R, int N)
{
    StageLayout s;
    s.offB = R * N * 4;
    s.offC = s.offB + kTokRows * N * 2;
    s.offX = s.offC + kTokRows * N * 2;
    s.offDt = s.offX + kTokRows * R * 2;
    s.offMeta = s.offDt + kTokRows * 8;
    s.bytes = (s.offMeta + static_cast<int>(sizeof(StageMeta)) + 127) / 128 * 128;
    const int fit = (static_cast<int>(kSmemBytes) - 128 - kOffStages) / s.bytes;
    s.count = fit < kMaxStages ? fit : kMaxStages;
    return s;
}

// Packed fp32x2 arithmetic (sm_100 and later): two independent fp32
// operations, each rounded to nearest even, in one instruction.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Sums each of v[0..K) over the L lanes (a power of two <= 32) of the aligned
// lane group: a butterfly whose steps first halve the values a lane holds (it
// keeps one half, its partner the other), then add the single value left.
// Afterwards this lane holds `count` totals, of value indices base .. base +
// count - 1; lanes that differ only in the bits of `dup` hold the same ones.
template <int K>
__device__ __forceinline__ void reduce_over_lanes(float (&v)[K], int L, int lane, int &base,
                                                  int &count, int &dup)
{
    base = 0;
    count = K;
    dup = 0;
    int o = L >> 1;
#pragma unroll
    for (int half = K / 2; half >= 1; half /= 2) {
        if (o == 0)
            break;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        if (upper)
            base += half;
        count = half;
        o >>= 1;
    }
    for (; o > 0; o >>= 1) {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        dup |= o;
    }
}

// NB (2, 4 or 8) consecutive bf16 values from shared memory, widened.
template <int NB>
__device__ __forceinline__ void load_bf16(const uint8_t *src, float (&out)[NB])
{
    if constexpr (NB == 8) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(src);
        const __nv_bfloat162 *v2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(v2[k]);
            out[2 * k] = f.x;
            out[2 * k + 1] = f.y;
        }
    } else if constexpr (NB == 4) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(src);
        const __nv_bfloat162 *v2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float2 f = __bfloat1622float2(v2[k]);
            out[2 * k] = f.x;
            out[2 * k + 1] = f.y;
        }
    } else {
        const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162 *>(src);
        const float2 f = __bfloat1622float2(v2);
        out[0] = f.x;
        out[1] = f.y;
    }
}

// One item on the consumer side: the thread's RB x NB block of the state
// tile (rows r0.., dstate columns n0..), the tokens' updates with y, and the
// final block back into the tile in the storage's element type.
template <int NB, int G>
__device__ __forceinline__ void consume(const ScanParams &p, const StageMeta &m, uint8_t *st,
                                        const StageLayout &sl, int es, int R, int N, int L,
                                        int lane, int r0, int n0, bool rows_ok, bool cols_ok)
{
    constexpr int RB = kElemsPerThread / NB;
    const float2 *sDtA = reinterpret_cast<const float2 *>(st + sl.offDt);
    const bool act = rows_ok && cols_ok;
    float s[RB][NB];
#pragma unroll
    for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int k = 0; k < NB; ++k)
            s[i][k] = 0.f;
    if (act && m.has_init) {
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            if (es == 4) {
#pragma unroll
                for (int k = 0; k < NB; k += 4) {
                    const float4 v =
                        *reinterpret_cast<const float4 *>(st + ((r0 + i) * N + n0 + k) * 4);
                    s[i][k] = v.x;
                    s[i][k + 1] = v.y;
                    s[i][k + 2] = v.z;
                    s[i][k + 3] = v.w;
                }
            } else {
                load_bf16<NB>(st + ((r0 + i) * N + n0) * 2, s[i]);
            }
        }
    }
    // tokens in groups of G: their updates are independent work for the
    // scheduler, and the group's G x RB row sums share one butterfly
    const __nv_bfloat16 *sX = reinterpret_cast<const __nv_bfloat16 *>(st + sl.offX);
    for (int tg = 0; tg < m.len; tg += G) {
        float part[G * RB];
#pragma unroll
        for (int u = 0; u < G; ++u) {
            const int t = tg + u;
#pragma unroll
            for (int i = 0; i < RB; ++i)
                part[u * RB + i] = 0.f;
            if (t < m.len) {
                const float2 da = sDtA[t];   // processed dt, exp(A dt)
                float xv[RB], b[NB], c[NB];
                if (rows_ok) {
                    load_bf16<RB>(st + sl.offX + (t * R + r0) * 2, xv);
                } else {
#pragma unroll
                    for (int i = 0; i < RB; ++i)
                        xv[i] = 0.f;
                }
                if (cols_ok) {
                    load_bf16<NB>(st + sl.offB + (t * N + n0) * 2, b);
                    load_bf16<NB>(st + sl.offC + (t * N + n0) * 2, c);
                } else {
#pragma unroll
                    for (int k = 0; k < NB; ++k)
                        b[k] = c[k] = 0.f;
                }
                // column pairs in packed fp32x2 instructions (the kernel is
                // bound by instruction issue on sequences of several tokens)
                const float2 dA2 = make_float2(da.y, da.y);
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    const float w = da.x * xv[i];
                    const float2 w2 = make_float2(w, w);
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < NB; k += 2) {
                        const float2 wb = fmul2(w2, make_float2(b[k], b[k + 1]));
                        const float2 sn = ffma2(make_float2(s[i][k], s[i][k + 1]), dA2, wb);
                        s[i][k] = sn.x;
                        s[i][k + 1] = sn.y;
                        acc = ffma2(make_float2(c[k], c[k + 1]), sn, acc);
                    }
                    part[u * RB + i] = acc.x + acc.y;
                }
            }
        }
        int base, count, dup;
        reduce_over_lanes<G * RB>(part, L, lane, base, count, dup);
        if (rows_ok && (lane & dup) == 0) {
            // one total per lane unless the row group has fewer lanes than values
            auto store = [&](int i, float v) {
                const int t = tg + (base + i) / RB, row = r0 + (base + i) % RB;
                if (t < m.len)
                    p.y[(static_cast<int64_t>(m.t0) + t) * p.y_ts +
                        static_cast<int64_t>(m.h) * p.P + m.row0 + row] =
                        __float2bfloat16_rn(v + m.Dh * __bfloat162float(sX[t * R + row]));
            };
            if (count == 1) {
                store(0, part[0]);
            } else {
#pragma unroll
                for (int i = 0; i < G * RB; ++i)
                    if (i < count)
                        store(i, part[i]);
            }
        }
    }
    if (act) {
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            if (es == 4) {
#pragma unroll
                for (int k = 0; k < NB; k += 4)
                    *reinterpret_cast<float4 *>(st + ((r0 + i) * N + n0 + k) * 4) =
                        make_float4(s[i][k], s[i][k + 1], s[i][k + 2], s[i][k + 3]);
            } else {
                uint32_t packed[NB / 2];
#pragma unroll
                for (int k = 0; k < NB / 2; ++k)
                    packed[k] = pack_bf16(s[i][2 * k], s[i][2 * k + 1]);
                if constexpr (NB == 8)
                    *reinterpret_cast<uint4 *>(st + ((r0 + i) * N + n0) * 2) =
                        make_uint4(packed[0], packed[1], packed[2], packed[3]);
                else
                    *reinterpret_cast<uint2 *>(st + ((r0 + i) * N + n0) * 2) =
                        make_uint2(packed[0], packed[1]);
            }
        }
    }
}

// 18 warps put 5 on two of the SM's four register-file quarters (16 K
// registers each), so 96 registers per thread is the most a launch can have
__global__ void __maxnreg__(96)
    short_scan_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, ScanParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBars);
    uint64_t *done = full + kMaxStages;
    uint64_t *empty = done + kMaxStages;
    volatile int32_t *s_failed = reinterpret_cast<volatile int32_t *>(smem + kOffFailed);

    const int P = p.P, N = p.N;
    const int R = tile_rows(P, N);
    const StageLayout sl = stage_layout(R, N);
    const int nst = sl.count;
    auto stage = [&](int s) { return smem + kOffStages + s * sl.bytes; };
    auto meta = [&](int s) { return reinterpret_cast<StageMeta *>(stage(s) + sl.offMeta); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            ptx::mbar_init(full + s, 32);
            ptx::mbar_init(done + s, kGroupWarps);
            ptx::mbar_init(empty + s, 1);
        }
        *s_failed = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();

    // the bookkeeping has checked query_start_loc and listed the short
    // sequences; only then is anything read or written
    pdl_wait();
    if (!p.hdr->valid)
        return;

    const int tph = P / R;                    // tiles per head
    const int per_seq = p.H * tph;
    const int n_items = p.hdr->n_short * per_seq;
    const int per_cta = (n_items + gridDim.x - 1) / gridDim.x;
    const int item_begin = blockIdx.x * per_cta;
    const int item_end = n_items < item_begin + per_cta ? n_items : item_begin + per_cta;
    const int es = (p.pool != nullptr && p.pool_bf16) ? 2 : 4;   // state element bytes
    const uint32_t tile_bytes = static_cast<uint32_t>(R * N * es);

    if (warp == kLoaderWarp) {
        // ------------------------------------------------------- loader warp
        const uint8_t *init_base = static_cast<const uint8_t *>(
            p.pool != nullptr ? static_cast<const void *>(p.pool)
                              : static_cast<const void *>(p.init_states));
        float2 *tab = reinterpret_cast<float2 *>(smem + kOffTab);   // [t][h - hb]: dt, exp(A dt)
        float *tabD = reinterpret_cast<float *>(smem + kOffTabD);
        if (lane == 0) {
            ptx::prefetch_tensormap(&tmX);
            ptx::prefetch_tensormap(&tmB);
            ptx::prefetch_tensormap(&tmC);
        }
        bool failed = false;
        int j = 0;   // items issued
        int cur_li = -1, hb = 0;
        SeqRec rec = {}, next_rec = {};
        if (item_begin < item_end)
            next_rec = p.short_list[item_begin / per_seq];
        // (sequence, head, tile) of the current item and its stage, stepped
        // along without divisions
        int li = item_begin / per_seq, h = (item_begin % per_seq) / tph, kt = item_begin % tph;
        int s = 0, round = 0;   // stage, and how often the stages have wrapped
        for (int item = item_begin; item < item_end; ++item, ++j) {
            if (item > item_begin) {
                if (++s == nst) {
                    s = 0;
                    ++round;
                }
                if (++kt == tph) {
                    kt = 0;
                    if (++h == p.H) {
                        h = 0;
                        ++li;
                    }
                }
            }
            const int row0 = kt * R;
            if (li != cur_li || h >= hb + kTabHeads) {
                if (li != cur_li) {
                    // the sequences of a CTA's range come in order: the record
                    // fetched ahead is this one's; fetch the following one
                    rec = next_rec;
                    cur_li = li;
                    if ((li + 1) * per_seq < item_end)
                        next_rec = p.short_list[li + 1];
                }
                // processed dt (as everywhere: softplus(dt + dt_bias)) and
                // exp(A dt) of the sequence's tokens for heads hb .. hb + 127;
                // a lane takes a head and loads all its tokens at once
                hb = h / kTabHeads * kTabHeads;
                const int nh = p.H - hb < kTabHeads ? p.H - hb : kTabHeads;
                __syncwarp();   // the previous table is no longer read
                for (int hh = lane; hh < nh; hh += 32) {
                    const float bias = p.dt_bias ? p.dt_bias[hb + hh] : 0.f;
                    const float a = p.A[hb + hh];
                    float raw[kShortLenMax];
#pragma unroll
                    for (int t = 0; t < kShortLenMax; ++t)
                        if (t < rec.len)
                            raw[t] = __bfloat162float(
                                p.dt[(static_cast<int64_t>(rec.t0) + t) * p.dt_ts + hb + hh]);
#pragma unroll
                    for (int t = 0; t < kShortLenMax; ++t)
                        if (t < rec.len) {
                            float v = raw[t];
                            if (p.dt_bias)
                                v += bias;
                            const float d = p.dt_softplus ? softplus_f32(v) : v;
                            tab[t * nh + hh] = make_float2(d, expf(a * d));
                        }
                    tabD[hh] = p.D ? p.D[hb + hh] : 0.f;
                }
                __syncwarp();
            }
            if (round > 0 && !ptx::mbar_wait(empty + s, (round - 1) & 1, kWaitTimeoutNs)) {
                failed = true;
                break;
            }
            uint8_t *st = stage(s);
            const int64_t tile_off = (static_cast<int64_t>(h) * P + row0) * N;
            const int nh = p.H - hb < kTabHeads ? p.H - hb : kTabHeads;
            if (lane < rec.len)
                reinterpret_cast<float2 *>(st + sl.offDt)[lane] = tab[lane * nh + (h - hb)];
            if (lane == 0) {
                StageMeta *m = meta(s);
                m->t0 = rec.t0;
                m->len = rec.len;
                m->h = h;
                m->row0 = row0;
                m->has_init = rec.init >= 0;
                m->Dh = tabD[h - hb];
                m->fin = rec.fin >= 0 ? rec.fin + tile_off : -1;
                // tensor copies move whole 8-token boxes (zeros past the end)
                const int boxes = (rec.len + kBox - 1) / kBox;
                const uint32_t bytes = (rec.init >= 0 ? tile_bytes : 0u) +
                                       static_cast<uint32_t>(boxes * kBox * (4 * N + 2 * R));
                ptx::mbar_arrive_expect_tx(full + s, bytes);
                if (rec.init >= 0)
                    ptx::bulk_load(st, init_base + (rec.init + tile_off) * es, tile_bytes, full + s);
                const int g = h / (p.H / p.G);
                for (int c = 0; c < boxes; ++c) {
                    const int t = rec.t0 + c * kBox;
                    ptx::tma_load_3d(st + sl.offB + c * kBox * N * 2, &tmB, full + s, 0, g, t);
                    ptx::tma_load_3d(st + sl.offC + c * kBox * N * 2, &tmC, full + s, 0, g, t);
                    ptx::tma_load_3d(st + sl.offX + c * kBox * R * 2, &tmX, full + s, h * P + row0,
                                     t, 0);
                }
            } else {
                ptx::mbar_arrive(full + s);
            }
        }
        if (failed) {
            if (lane == 0)
                record_error(p.hdr, kErrTimeout);
            *s_failed = 1;
            // bounded waits for the copies still landing in the stages
            for (int k = j - nst > 0 ? j - nst : 0; k < j; ++k)
                ptx::mbar_wait(full + k % nst, (k / nst) & 1, kWaitTimeoutNs);
        }
        return;
    }

    if (warp == kStorerWarp) {
        // ------------------------------------------------------- storer warp
        uint8_t *fin_base = static_cast<uint8_t *>(
            p.pool != nullptr ? p.pool : static_cast<void *>(p.final_states));
        int k = 0, s = 0, s_lag = 0;
        uint32_t ph = 0;
        for (int item = item_begin; item < item_end; ++item, ++k) {
            if (!ptx::mbar_wait(done + s, ph, kWaitTimeoutNs)) {
                if (lane == 0)
                    record_error(p.hdr, kErrTimeout);
                *s_failed = 1;
                break;
            }
            if (lane == 0) {
                const StageMeta *m = meta(s);
                if (m->fin >= 0)
                    ptx::bulk_store(fin_base + m->fin * es, stage(s), tile_bytes);
                ptx::bulk_commit_group();   // one group per item, empty without a store
                // the stores of items up to k - kStoreLag have read their stages
                ptx::bulk_wait_group_read<kStoreLag>();
                if (k >= kStoreLag)
                    ptx::mbar_arrive(empty + s_lag);
            }
            if (k >= kStoreLag && ++s_lag == nst)
                s_lag = 0;
            if (++s == nst) {
                s = 0;
                ph ^= 1u;
            }
            __syncwarp();
        }
        if (lane == 0)
            ptx::bulk_wait_group0();
        return;
    }

    // ------------------------------------------------------- consumer warps
    // NB dstate columns per thread (4, or 8 when more than 32 lanes of 4 would
    // be needed), RB = 16 / NB rows; L lanes share a row group (<= 32)
    const int Npad = pow2_at_least(N);
    const int NB = Npad > 128 ? 8 : 4;
    const int RB = kElemsPerThread / NB;
    const int L = Npad / NB;
    // group `grp` takes every kConsumerGroups-th item, starting with its own
    const int grp = warp / kGroupWarps, gtid = tid % kConsumers;
    const int lr = gtid % L, r0 = (gtid / L) * RB, n0 = lr * NB;
    const bool rows_ok = r0 < R, cols_ok = n0 < N;
    int s = grp;
    uint32_t ph = 0;
    for (int item = item_begin + grp; item < item_end; item += kConsumerGroups) {
        if (*s_failed || !ptx::mbar_wait(full + s, ph, kWaitTimeoutNs)) {
            record_error(p.hdr, kErrTimeout);
            break;
        }
        uint8_t *st = stage(s);
        const StageMeta m = *meta(s);
        // one token (a decode step) needs no token groups
        if (NB == 8) {
            if (m.len <= 1)
                consume<8, 1>(p, m, st, sl, es, R, N, L, lane, r0, n0, rows_ok, cols_ok);
            else
                consume<8, kGroup>(p, m, st, sl, es, R, N, L, lane, r0, n0, rows_ok, cols_ok);
        } else {
            if (m.len <= 1)
                consume<4, 1>(p, m, st, sl, es, R, N, L, lane, r0, n0, rows_ok, cols_ok);
            else
                consume<4, kGroup>(p, m, st, sl, es, R, N, L, lane, r0, n0, rows_ok, cols_ok);
        }
        // the storer's bulk store reads the tile through the async proxy; one
        // arrival per warp once all its lanes have written
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            ptx::mbar_arrive(done + s);
        s += kConsumerGroups;
        if (s >= nst) {
            s -= nst;
            ph ^= 1u;
        }
    }
}

SmemOptIn s_smem_configured;

}  // namespace

int short_scan_tile_rows(int P, int N) { return tile_rows(P, N); }

cudaError_t launch_short_scan(const ScanParams &p, const ShortScanMaps &maps, cudaStream_t stream,
                              bool programmatic)
{
    static_assert(kSmemBytes <= kMaxSmemPerBlock, "stages exceed shared memory");
    // the storer frees a stage kStoreLag items late: more stages than that
    // (at least 6 fit for every supported dstate)
    if (stage_layout(tile_rows(p.P, p.N), p.N).count <= kStoreLag)
        return cudaErrorInvalidConfiguration;
    cudaError_t e = ensure_max_smem(reinterpret_cast<const void *>(short_scan_kernel), s_smem_configured);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    // a persistent grid, one CTA per SM (fewer for small batches), over the
    // tiles of the short sequences the bookkeeping listed
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t items =
        static_cast<int64_t>(p.batch) * p.H * (p.P / tile_rows(p.P, p.N));
    cfg.gridDim = dim3(static_cast<unsigned>(items < sms ? items : sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, short_scan_kernel, maps.X, maps.B, maps.C, p);
}

}  // namespace ssd
