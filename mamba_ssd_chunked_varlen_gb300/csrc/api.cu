// C ABI of the scan (declared in include/ssd_scan.h): argument checks,
// workspace carving, TMA descriptor encoding and the stage launches on the
// caller's stream.  No host synchronisation, no allocation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/ssd_scan.h"
#include "kernels.cuh"

namespace {

using ssd::ScanParams;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D bf16 tensor map with a {b0, b1, b2} box and no swizzle (rows land
// packed in shared memory).  Elements outside the tensor read as zero.
bool make_map_plain(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
                    uint32_t b2)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor map with a {64, b1, b2} box and 128-byte swizzle.  Elements
// outside the tensor read as zero.
bool make_map_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b1, uint32_t b2)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {64, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Limit of the deliberate never-completed wait (ssd_scan_varlen_test_stall);
// 0 outside the tests of the bounded-wait path.
std::atomic<uint32_t> g_test_stall_ns{0};

// Whether a call may hold sequences of at most kShortLenMax tokens (then the
// short-sequence kernel runs): a batch of several sequences, or one sequence
// that short.  A single longer sequence needs no such launch.
bool short_path(int64_t total_len, int32_t batch)
{
    return batch > 1 || total_len <= ssd::kShortLenMax;
}

// Sequences of at most this many tokens go to the short-sequence kernel.
int32_t short_len_of(int64_t total_len, int32_t batch)
{
    return short_path(total_len, batch) ? ssd::kShortLenMax : 0;
}

ssd_status_t check_sizes(int64_t T, int32_t batch, int32_t H, int32_t P, int32_t G, int32_t N,
                         int32_t Q)
{
    if (T < 0 || batch < 0 || H <= 0 || P <= 0 || G <= 0 || N <= 0 || Q <= 0)
        return SSD_ERR_INVALID_ARG;
    if (H % G != 0)
        return SSD_ERR_INVALID_ARG;
    if (N > SSD_MAX_DSTATE)
        return SSD_ERR_UNSUPPORTED;
    if ((P != 16 && P != 32 && P != 64 && P != 128) || N % 16 != 0 || N < 16)
        return SSD_ERR_UNSUPPORTED;
    if (Q != 64 && Q != 128 && Q != 256)
        return SSD_ERR_UNSUPPORTED;
    if (T > INT32_MAX / 2 || static_cast<int64_t>(batch) > INT32_MAX / 2)
        return SSD_ERR_UNSUPPORTED;
    const ssd::K1Config k1 = ssd::chunk_state_config(H, G, P, N);
    const ssd::K3Config k3 = ssd::chunk_scan_config(H, G, P, N);
    const ssd::WalkConfig kw = ssd::state_walk_config(H, G, P, N, batch > 0 ? batch : 1, 1);
    if (k1.HB == 0 || k3.HB == 0)
        return SSD_ERR_UNSUPPORTED;
    if (k1.smem > static_cast<size_t>(ssd::kMaxSmemPerBlock) ||
        k3.smem > static_cast<size_t>(ssd::kMaxSmemPerBlock) ||
        kw.smem > static_cast<size_t>(ssd::kMaxSmemPerBlock))
        return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

}  // namespace

extern "C" {

const char *ssd_status_string(ssd_status_t s)
{
    switch (s) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARG: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "unsupported size";
    case SSD_ERR_WORKSPACE: return "workspace missing or too small";
    case SSD_ERR_CUDA: return "CUDA error";
    case SSD_ERR_DEVICE: return "device-side error flag set";
    case SSD_ERR_TOO_LARGE: return "sizes need more scratch than the built-in no-allocation buffer";
    }
    return "unknown status";
}

size_t ssd_scan_varlen_workspace_size(int64_t total_len, int32_t batch, int32_t nheads,
                                      int32_t head_dim, int32_t ngroups, int32_t dstate,
                                      int32_t chunk_size)
{
    if (check_sizes(total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size) != SSD_OK)
        return 0;
    return ssd::ws_layout(total_len, batch, nheads, head_dim, dstate,
                          ssd::block_tokens(chunk_size), short_len_of(total_len, batch)).total;
}

int32_t ssd_scan_varlen_short_threshold(int64_t total_len, int32_t batch)
{
    return batch > 0 ? short_len_of(total_len, batch) : 0;
}

int32_t ssd_scan_varlen_fused_walk(int64_t total_len, int32_t batch, int32_t nheads,
                                   int32_t head_dim, int32_t ngroups, int32_t dstate,
                                   int32_t chunk_size)
{
    if (batch <= 0 ||
        check_sizes(total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size) != SSD_OK)
        return 0;
    return ssd::use_state_walk(total_len, batch, nheads, ngroups, head_dim, dstate,
                               ssd::block_tokens(chunk_size))
               ? 1
               : 0;
}

int32_t ssd_scan_varlen_num_launches(int64_t total_len, int32_t batch, int32_t nheads,
                                     int32_t head_dim, int32_t ngroups, int32_t dstate,
                                     int32_t chunk_size)
{
    if (batch <= 0)
        return 0;
    const int walk = ssd_scan_varlen_fused_walk(total_len, batch, nheads, head_dim, ngroups,
                                                dstate, chunk_size);
    const bool table =
        ssd::use_block_table(total_len, batch, nheads, ngroups, head_dim, dstate,
                             ssd::block_tokens(chunk_size), short_len_of(total_len, batch));
    return (walk ? 1 : 2) + (total_len > 0 ? 1 : 0) + (short_path(total_len, batch) ? 1 : 0) +
           (table ? 1 : 0);
}

}  // extern "C"

namespace ssd {

ssd_status_t scan_impl(void *y, const void *x, const void *dt, const float *A, const void *B,
                       const void *C, const float *D, const float *dt_bias, const StateIO &io,
                       const int32_t *query_start_loc, const uint8_t *has_initial_state,
                       int64_t total_len, int32_t batch, int32_t nheads, int32_t head_dim,
                       int32_t ngroups, int32_t dstate, int32_t chunk_size, int32_t dt_softplus,
                       void *workspace, size_t workspace_bytes, ssd_stream_t stream_,
                       void *const *events, const TokenStrides *strides, bool launch)
{
    const ssd_status_t sz =
        check_sizes(total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size);
    if (sz != SSD_OK)
        return sz;
    const bool in_place = io.pool != nullptr;
    if (in_place && io.max_slots < 0)
        return SSD_ERR_INVALID_ARG;
    if (batch == 0)
        return SSD_OK;
    if (!query_start_loc || !A)
        return SSD_ERR_INVALID_ARG;
    if (in_place ? !io.cache_indices : !io.final_states)
        return SSD_ERR_INVALID_ARG;
    if (total_len > 0 && (!y || !x || !dt || !B || !C))
        return SSD_ERR_INVALID_ARG;
    if (total_len > 0 && (!aligned16(y) || !aligned16(x) || !aligned16(B) || !aligned16(C)))
        return SSD_ERR_INVALID_ARG;
    if (!aligned16(io.pool) || !aligned16(io.initial_states) || !aligned16(io.final_states))
        return SSD_ERR_INVALID_ARG;
    // token strides: at least the row of one token; TMA reads x, B, C with row
    // pitches that are multiples of 16 bytes, and y rows are stored 16 bytes at a time
    const int64_t HP = static_cast<int64_t>(nheads) * head_dim, GN = static_cast<int64_t>(ngroups) * dstate;
    const TokenStrides ts{strides && strides->x ? strides->x : HP,
                          strides && strides->dt ? strides->dt : nheads,
                          strides && strides->B ? strides->B : GN,
                          strides && strides->C ? strides->C : GN,
                          strides && strides->y ? strides->y : HP};
    if (ts.x < HP || ts.dt < nheads || ts.B < GN || ts.C < GN || ts.y < HP)
        return SSD_ERR_INVALID_ARG;
    if (ts.x % 8 || ts.B % 8 || ts.C % 8 || ts.y % 8)
        return SSD_ERR_INVALID_ARG;
    const int32_t Qb = ssd::block_tokens(chunk_size);
    const ssd::WsLayout L =
        ssd::ws_layout(total_len, batch, nheads, head_dim, dstate, Qb, short_len_of(total_len, batch));
    if (!workspace || workspace_bytes < L.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return SSD_ERR_WORKSPACE;
    if (L.max_chunks * nheads > INT32_MAX)
        return SSD_ERR_UNSUPPORTED;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    ScanParams p;
    std::memset(&p, 0, sizeof p);
    p.y = static_cast<__nv_bfloat16 *>(y);
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.dt = static_cast<const __nv_bfloat16 *>(dt);
    p.B = static_cast<const __nv_bfloat16 *>(B);
    p.C = static_cast<const __nv_bfloat16 *>(C);
    p.A = A;
    p.D = D;
    p.dt_bias = dt_bias;
    p.pool = io.pool;
    p.pool_bf16 = io.pool_bf16;
    p.cache_idx = io.cache_indices;
    p.max_slots = io.max_slots;
    p.init_states = io.initial_states;
    p.final_states = io.final_states;
    p.qsl = query_start_loc;
    p.has_init = has_initial_state;
    p.T = total_len;
    p.x_ts = ts.x;
    p.dt_ts = ts.dt;
    p.B_ts = ts.B;
    p.C_ts = ts.C;
    p.y_ts = ts.y;
    p.batch = batch;
    p.H = nheads;
    p.P = head_dim;
    p.G = ngroups;
    p.N = dstate;
    p.Q = Qb;
    p.dt_softplus = dt_softplus ? 1 : 0;
    p.short_len = short_len_of(total_len, batch);
    // calls of long sequences with many heads take the fused walk (the block
    // states stay on chip); the others the split chunk-state / state-passing pair
    const bool walk = ssd::use_state_walk(total_len, batch, nheads, ngroups, head_dim, dstate, Qb);
    p.finish_single = (!walk && batch > 1) ? 1 : 0;
    p.max_chunks = static_cast<int32_t>(L.max_chunks);
    p.test_stall_ns = g_test_stall_ns.load(std::memory_order_relaxed);
    p.hdr = reinterpret_cast<ssd::WsHeader *>(ws + L.header);
    p.seq_first = reinterpret_cast<int32_t *>(ws + L.seq_first);
    p.short_list = reinterpret_cast<ssd::SeqRec *>(ws + L.short_list);
    p.long_list = reinterpret_cast<ssd::SeqRec *>(ws + L.long_list);
    p.table = ssd::use_block_table(total_len, batch, nheads, ngroups, head_dim, dstate, Qb,
                                   p.short_len)
                  ? reinterpret_cast<ssd::BlockEntry *>(ws + L.table)
                  : nullptr;
    p.decay = reinterpret_cast<float *>(ws + L.decay);
    p.schunk = reinterpret_cast<__half *>(ws + L.schunk);
    p.sexp = reinterpret_cast<int8_t *>(ws + L.sexp);
    p.sprev = reinterpret_cast<__nv_bfloat16 *>(ws + L.sprev);

    ssd::ChunkStateMaps m1;
    ssd::StateWalkMaps mw;
    ssd::ChunkScanMaps m3;
    ssd::ShortScanMaps ms;
    std::memset(&m1, 0, sizeof m1);  // with total_len == 0 no kernel reads a map
    std::memset(&mw, 0, sizeof mw);
    std::memset(&m3, 0, sizeof m3);
    std::memset(&ms, 0, sizeof ms);
    if (total_len > 0) {
        const uint64_t T = static_cast<uint64_t>(total_len);
        const uint64_t H = nheads, P = head_dim, G = ngroups, N = dstate;
        const uint64_t xs = ts.x * 2, bs = ts.B * 2, cs = ts.C * 2;   // token pitches, bytes
        bool ok = make_map_3d(&m1.B, B, N, G, T, N * 2, bs, 1, 64) &&
                  make_map_3d(&m1.X, x, H * P, T, 1, xs, xs * T, 64, 1) &&
                  make_map_3d(&m3.B, B, N, G, T, N * 2, bs, 1, 64) &&
                  make_map_3d(&m3.C, C, N, G, T, N * 2, cs, 1, 64) &&
                  make_map_3d(&m3.X, x, H * P, T, 1, xs, xs * T, 64, 1) &&
                  make_map_3d(&m3.Sprev, p.sprev, N, P, static_cast<uint64_t>(L.max_chunks) * H,
                              N * 2, P * N * 2, 64, 1);
        if (ok && walk) {
            // dt by TMA when its base and row pitch are 16-byte aligned
            mw.B = m1.B;
            mw.X = m1.X;
            mw.dt_tma = aligned16(dt) && ts.dt % 8 == 0 &&
                        make_map_plain(&mw.Dt, dt, H, T, 1, ts.dt * 2, ts.dt * 2 * T, 16, 64, 1);
        }
        if (ok && p.short_len > 0) {
            const uint32_t R = static_cast<uint32_t>(ssd::short_scan_tile_rows(head_dim, dstate));
            ok = make_map_plain(&ms.X, x, H * P, T, 1, xs, xs * T, R, 8, 1) &&
                 make_map_plain(&ms.B, B, N, G, T, N * 2, bs, static_cast<uint32_t>(N), 1, 8) &&
                 make_map_plain(&ms.C, C, N, G, T, N * 2, cs, static_cast<uint32_t>(N), 1, 8);
        }
        if (!ok)
            return SSD_ERR_CUDA;
    }
    if (!launch)
        return SSD_OK;

    // Stage events (profiled entry point): before the first launch and after
    // each launch.  Between launches they also end the programmatic overlap.
    auto mark = [&](int k) {
        return events == nullptr ||
               cudaEventRecord(static_cast<cudaEvent_t>(events[k]), stream) == cudaSuccess;
    };
    const bool pdl = events == nullptr;
    // large batches: the block map first, the chunk-state kernel (or the walk)
    // its dependent; with the walk the state-passing stage has no launch
    const bool mapped = p.table != nullptr;
    if (!mark(0) || (mapped && ssd::launch_block_map(p, stream) != cudaSuccess))
        return SSD_ERR_CUDA;
    if ((walk ? ssd::launch_state_walk(p, mw, stream, mapped && pdl)
              : ssd::launch_chunk_state(p, m1, stream, mapped && pdl)) != cudaSuccess ||
        !mark(1))
        return SSD_ERR_CUDA;
    if ((!walk && ssd::launch_state_passing(p, stream, pdl) != cudaSuccess) || !mark(2))
        return SSD_ERR_CUDA;
    if (total_len > 0 && ssd::launch_chunk_scan(p, m3, stream, pdl) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (!mark(3))
        return SSD_ERR_CUDA;
    if (p.short_len > 0 && ssd::launch_short_scan(p, ms, stream, pdl) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (!mark(4))
        return SSD_ERR_CUDA;
    return SSD_OK;
}

}  // namespace ssd

extern "C" {

ssd_status_t ssd_scan_varlen_fwd(void *y, const void *x, const void *dt, const float *A,
                                 const void *B, const void *C, const float *D,
                                 const float *dt_bias, float *ssm_pool,
                                 const int32_t *query_start_loc,
                                 const uint8_t *has_initial_state, const uint32_t *cache_indices,
                                 int64_t total_len, int32_t batch, int32_t nheads,
                                 int32_t head_dim, int32_t ngroups, int32_t dstate,
                                 int64_t max_slots, int32_t chunk_size, int32_t dt_softplus,
                                 void *workspace, size_t workspace_bytes, ssd_stream_t stream)
{
    const ssd::StateIO io{ssm_pool, cache_indices, max_slots, nullptr, nullptr, 0};
    if (!ssm_pool && batch > 0)
        return SSD_ERR_INVALID_ARG;
    return ssd::scan_impl(y, x, dt, A, B, C, D, dt_bias, io, query_start_loc, has_initial_state,
                          total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size,
                          dt_softplus, workspace, workspace_bytes, stream, nullptr);
}

ssd_status_t ssd_scan_varlen_fwd_bf16_pool(void *y, const void *x, const void *dt, const float *A,
                                           const void *B, const void *C, const float *D,
                                           const float *dt_bias, void *ssm_pool,
                                           const int32_t *query_start_loc,
                                           const uint8_t *has_initial_state,
                                           const uint32_t *cache_indices, int64_t total_len,
                                           int32_t batch, int32_t nheads, int32_t head_dim,
                                           int32_t ngroups, int32_t dstate, int64_t max_slots,
                                           int32_t chunk_size, int32_t dt_softplus,
                                           void *workspace, size_t workspace_bytes,
                                           ssd_stream_t stream)
{
    const ssd::StateIO io{ssm_pool, cache_indices, max_slots, nullptr, nullptr, 1};
    if (!ssm_pool && batch > 0)
        return SSD_ERR_INVALID_ARG;
    return ssd::scan_impl(y, x, dt, A, B, C, D, dt_bias, io, query_start_loc, has_initial_state,
                          total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size,
                          dt_softplus, workspace, workspace_bytes, stream, nullptr);
}

ssd_status_t ssd_scan_varlen_fwd_strided(void *y, const void *x, const void *dt, const float *A,
                                         const void *B, const void *C, const float *D,
                                         const float *dt_bias, float *ssm_pool,
                                         const int32_t *query_start_loc,
                                         const uint8_t *has_initial_state,
                                         const uint32_t *cache_indices, int64_t total_len,
                                         int32_t batch, int32_t nheads, int32_t head_dim,
                                         int32_t ngroups, int32_t dstate, int64_t max_slots,
                                         int32_t chunk_size, int32_t dt_softplus,
                                         const ssd_token_strides_t *strides, void *workspace,
                                         size_t workspace_bytes, ssd_stream_t stream)
{
    const ssd::StateIO io{ssm_pool, cache_indices, max_slots, nullptr, nullptr, 0};
    if (!ssm_pool && batch > 0)
        return SSD_ERR_INVALID_ARG;
    ssd::TokenStrides ts{0, 0, 0, 0, 0};
    if (strides)
        ts = ssd::TokenStrides{strides->x, strides->dt, strides->B, strides->C, strides->y};
    return ssd::scan_impl(y, x, dt, A, B, C, D, dt_bias, io, query_start_loc, has_initial_state,
                          total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size,
                          dt_softplus, workspace, workspace_bytes, stream, nullptr, &ts);
}

ssd_status_t ssd_scan_varlen_fwd_states(void *y, const void *x, const void *dt, const float *A,
                                        const void *B, const void *C, const float *D,
                                        const float *dt_bias, const float *initial_states,
                                        const uint8_t *has_initial_state, float *final_states,
                                        const int32_t *query_start_loc, int64_t total_len,
                                        int32_t batch, int32_t nheads, int32_t head_dim,
                                        int32_t ngroups, int32_t dstate, int32_t chunk_size,
                                        int32_t dt_softplus, void *workspace,
                                        size_t workspace_bytes, ssd_stream_t stream)
{
    const ssd::StateIO io{nullptr, nullptr, 0, initial_states, final_states, 0};
    return ssd::scan_impl(y, x, dt, A, B, C, D, dt_bias, io, query_start_loc, has_initial_state,
                          total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size,
                          dt_softplus, workspace, workspace_bytes, stream, nullptr);
}

ssd_status_t ssd_scan_varlen_fwd_profiled(
    void *y, const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, const float *dt_bias, float *ssm_pool, const int32_t *query_start_loc,
    const uint8_t *has_initial_state, const uint32_t *cache_indices, int64_t total_len,
    int32_t batch, int32_t nheads, int32_t head_dim, int32_t ngroups, int32_t dstate,
    int64_t max_slots, int32_t chunk_size, int32_t dt_softplus, void *workspace,
    size_t workspace_bytes, ssd_stream_t stream, void *const *events)
{
    if (!events)
        return SSD_ERR_INVALID_ARG;
    for (int k = 0; k < 5; ++k)
        if (!events[k])
            return SSD_ERR_INVALID_ARG;
    const ssd::StateIO io{ssm_pool, cache_indices, max_slots, nullptr, nullptr, 0};
    if (!ssm_pool && batch > 0)
        return SSD_ERR_INVALID_ARG;
    return ssd::scan_impl(y, x, dt, A, B, C, D, dt_bias, io, query_start_loc, has_initial_state,
                          total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size,
                          dt_softplus, workspace, workspace_bytes, stream, events);
}

void ssd_scan_varlen_test_stall(uint32_t limit_ns) { g_test_stall_ns.store(limit_ns); }

ssd_status_t ssd_scan_varlen_read_errors(const void *workspace, ssd_stream_t stream_,
                                         uint32_t *flags)
{
    if (!workspace || !flags)
        return SSD_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    *flags = v;
    return v ? SSD_ERR_DEVICE : SSD_OK;
}

}  // extern "C"
