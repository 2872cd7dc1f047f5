// End-to-end call with the per-step tensors in host memory (declared in
// include/ssd_scan.h): the token range is cut into pieces whose host->device
// copies, scans and device->host copies of y overlap on three streams.
//
// A piece is a token range [a, e).  Its sequences are the parts of the
// call's sequences that fall inside it, in batch order; a part that does not
// start at its sequence's first token continues from the sequence's slot
// (which the previous piece's part wrote), so the pieces together compute
// the state recurrence of the whole call.  Cuts are placed on block
// boundaries of the sequence they fall in (multiples of the block length
// from its start): every block is the block the single call would form.
//
// Host code only; the scan of each piece is the regular launch sequence.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/ssd_scan.h"
#include "kernels.cuh"

namespace {

constexpr int kMaxPieces = SSD_HOST_MAX_PIECES;
constexpr int kMaxDevices = 64;
constexpr uint32_t kDirMagic = 0x53534448u;   // marks a host-call workspace directory

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Directory at the start of the workspace: where each piece's scan
// workspace lies (for ssd_scan_varlen_host_read_errors).
struct Directory {
    uint32_t magic;
    uint32_t pieces;
    uint64_t scan_ws[kMaxPieces];
};
static_assert(sizeof(Directory) <= 256, "directory must fit its 256-byte region");

// query_start_loc from 0, never decreasing, ending at total_len.
bool qsl_valid(const int32_t *qsl, int64_t T, int32_t batch)
{
    if (!qsl || batch < 0 || T < 0 || qsl[0] != 0 || qsl[batch] != T)
        return false;
    for (int32_t b = 0; b < batch; ++b)
        if (qsl[b + 1] < qsl[b])
            return false;
    return true;
}

// Cut positions (strictly increasing, inside (0, T)).  The k-th of n - 1
// target positions k T / n moves to the nearest block boundary of the
// sequence that holds it (or that sequence's end).
std::vector<int64_t> plan_cuts(const int32_t *qsl, int64_t T, int32_t batch, int Qb, int n)
{
    std::vector<int64_t> cuts;
    int64_t prev = 0;
    int32_t b = 0;
    for (int k = 1; k < n; ++k) {
        const int64_t t = T * k / n;
        while (b < batch && qsl[b + 1] <= t)
            ++b;
        if (b >= batch)
            break;
        const int64_t s = qsl[b], f = qsl[b + 1];
        int64_t c = s + (t - s + Qb / 2) / Qb * Qb;
        if (c > f)
            c = f;
        if (c <= prev || c >= T)
            continue;
        cuts.push_back(c);
        prev = c;
    }
    return cuts;
}

// Pieces when the caller leaves the choice: one per ~6 MiB of input.  A
// host<->device copy costs ~5 us beyond its bytes (measured on GB300 over
// the host link at ~190 GB/s per direction), and a piece adds four input
// copies and one output copy, so pieces much smaller than that lose more
// to the copies' own cost than the overlap gains.
int auto_pieces(int64_t T, int32_t H, int32_t P, int32_t G, int32_t N)
{
    const int64_t in_bytes = T * (static_cast<int64_t>(H) * P * 2 + H * 2 +
                                  static_cast<int64_t>(G) * N * 4);
    const int64_t n = in_bytes / (int64_t(6) << 20);
    return n < 1 ? 1 : (n > kMaxPieces ? kMaxPieces : static_cast<int>(n));
}

// One piece: its token range and its sequences' local arguments.
struct Piece {
    int64_t a = 0, e = 0;
    std::vector<int32_t> qsl;      // local query_start_loc (b_k + 1)
    std::vector<uint32_t> cidx;    // slots
    std::vector<uint8_t> hinit;    // initial-state flags (1 for continuations)
    size_t meta_off = 0, ws_off = 0, ws_bytes = 0;
    int32_t batch() const { return static_cast<int32_t>(cidx.size()); }
};

struct Plan {
    std::vector<Piece> pieces;
    size_t meta_end = 0;   // the directory and the pieces' small arrays: [0, meta_end)
    size_t x_off = 0, dt_off = 0, B_off = 0, C_off = 0, y_off = 0, total = 0;
};

// The pieces of a call and the workspace layout: the directory and every
// piece's small arrays (one copy from the host), the device copies of x, dt,
// B, C and y, then per piece its scan workspace.
// Returns false when a piece's sizes are unsupported.
bool make_plan(Plan &pl, const int32_t *qsl, const uint8_t *hinit, const uint32_t *cidx,
               int64_t T, int32_t batch, int32_t H, int32_t P, int32_t G, int32_t N, int32_t Q,
               int n_req)
{
    const int Qb = ssd::block_tokens(Q);
    const int n = n_req > 0 ? (n_req < kMaxPieces ? n_req : kMaxPieces)
                            : auto_pieces(T, H, P, G, N);
    const std::vector<int64_t> cuts = plan_cuts(qsl, T, batch, Qb, n);
    const int np = static_cast<int>(cuts.size()) + 1;
    pl.pieces.assign(np, Piece());
    for (int k = 0; k < np; ++k) {
        Piece &pc = pl.pieces[k];
        pc.a = k == 0 ? 0 : cuts[k - 1];
        pc.e = k == np - 1 ? T : cuts[k];
        pc.qsl.push_back(0);
        for (int32_t b = 0; b < batch; ++b) {
            const int64_t s = qsl[b], f = qsl[b + 1];
            bool in;
            int64_t lo, hi;
            if (s == f) {
                // an empty sequence belongs to the piece its position starts
                // (the last piece when it sits at total_len)
                in = (s >= pc.a && s < pc.e) || (s == T && k == np - 1);
                lo = hi = s;
            } else {
                lo = s > pc.a ? s : pc.a;
                hi = f < pc.e ? f : pc.e;
                in = lo < hi;
            }
            if (!in)
                continue;
            pc.qsl.push_back(static_cast<int32_t>(hi - pc.a));
            pc.cidx.push_back(cidx ? cidx[b] : 0u);
            pc.hinit.push_back(lo > s ? 1 : (hinit && hinit[b] ? 1 : 0));
        }
    }
    size_t off = 256;   // directory
    for (Piece &pc : pl.pieces) {
        const size_t b = pc.cidx.size();
        pc.meta_off = off;
        off = (off + (b + 1) * 4 + b * 4 + b + 15) & ~size_t(15);
    }
    pl.meta_end = off;
    off = align256(off);
    const size_t HP = static_cast<size_t>(H) * P, GN = static_cast<size_t>(G) * N;
    const size_t Tz = static_cast<size_t>(T);
    pl.x_off = off;
    off = align256(off + Tz * HP * 2);
    pl.dt_off = off;
    off = align256(off + Tz * H * 2);
    pl.B_off = off;
    off = align256(off + Tz * GN * 2);
    pl.C_off = off;
    off = align256(off + Tz * GN * 2);
    pl.y_off = off;
    off = align256(off + Tz * HP * 2);
    for (Piece &pc : pl.pieces) {
        pc.ws_bytes = ssd_scan_varlen_workspace_size(pc.e - pc.a, pc.batch(), H, P, G, N, Q);
        if (pc.ws_bytes == 0)
            return false;
        pc.ws_off = off;
        off = align256(off + pc.ws_bytes);
    }
    pl.total = off;
    return true;
}

// The internal copy streams and events of one device, created on first use
// and kept for the life of the process, and a ring of pinned host buffers
// from which the small arrays are copied (a copy from pageable memory may
// block the host until its stream reaches it, which would hold back the
// launches queued after it).  A ring slot is reused once its last copy is
// done.
constexpr int kRing = 4;
struct DeviceStreams {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[kMaxPieces] = {}, scan_done[kMaxPieces] = {};
    uint8_t *stage[kRing] = {};
    size_t stage_bytes[kRing] = {};
    cudaEvent_t stage_done[kRing] = {};
    bool stage_used[kRing] = {};
    unsigned next = 0;
};

std::mutex g_mutex;   // guards g_dev and serialises the enqueue of calls
DeviceStreams g_dev[kMaxDevices];

cudaError_t device_streams(DeviceStreams **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    DeviceStreams &d = g_dev[dev];
    if (!d.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&d.h2d, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&d.d2h, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&d.start, ef)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&d.end, ef)) != cudaSuccess)
            return e;
        for (int k = 0; k < kMaxPieces; ++k)
            if ((e = cudaEventCreateWithFlags(&d.in_done[k], ef)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&d.scan_done[k], ef)) != cudaSuccess)
                return e;
        for (int k = 0; k < kRing; ++k)
            if ((e = cudaEventCreateWithFlags(&d.stage_done[k], ef)) != cudaSuccess)
                return e;
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

}  // namespace

extern "C" {

int32_t ssd_scan_varlen_host_plan(const int32_t *query_start_loc_host, int64_t total_len,
                                  int32_t batch, int32_t nheads, int32_t head_dim,
                                  int32_t ngroups, int32_t dstate, int32_t chunk_size,
                                  int32_t pieces, int64_t *cuts_out)
{
    if (!qsl_valid(query_start_loc_host, total_len, batch) || !cuts_out ||
        (chunk_size != 64 && chunk_size != 128 && chunk_size != 256) || nheads <= 0 ||
        head_dim <= 0 || ngroups <= 0 || dstate <= 0)
        return -1;
    const int n = pieces > 0 ? (pieces < kMaxPieces ? pieces : kMaxPieces)
                             : auto_pieces(total_len, nheads, head_dim, ngroups, dstate);
    const std::vector<int64_t> cuts = plan_cuts(query_start_loc_host, total_len, batch,
                                                ssd::block_tokens(chunk_size), n);
    for (size_t i = 0; i < cuts.size(); ++i)
        cuts_out[i] = cuts[i];
    return static_cast<int32_t>(cuts.size()) + 1;
}

size_t ssd_scan_varlen_host_workspace_size(const int32_t *query_start_loc_host,
                                           int64_t total_len, int32_t batch, int32_t nheads,
                                           int32_t head_dim, int32_t ngroups, int32_t dstate,
                                           int32_t chunk_size, int32_t pieces)
{
    if (ssd_scan_varlen_workspace_size(total_len, batch, nheads, head_dim, ngroups, dstate,
                                       chunk_size) == 0 ||
        !qsl_valid(query_start_loc_host, total_len, batch))
        return 0;
    Plan pl;
    if (!make_plan(pl, query_start_loc_host, nullptr, nullptr, total_len, batch, nheads,
                   head_dim, ngroups, dstate, chunk_size, pieces))
        return 0;
    return pl.total;
}

ssd_status_t ssd_scan_varlen_fwd_host(
    void *y_host, const void *x_host, const void *dt_host, const float *A, const void *B_host,
    const void *C_host, const float *D, const float *dt_bias, float *ssm_pool,
    const int32_t *query_start_loc_host, const uint8_t *has_initial_state_host,
    const uint32_t *cache_indices_host, int64_t total_len, int32_t batch, int32_t nheads,
    int32_t head_dim, int32_t ngroups, int32_t dstate, int64_t max_slots, int32_t chunk_size,
    int32_t dt_softplus, int32_t pieces, void *workspace, size_t workspace_bytes,
    ssd_stream_t stream_)
{
    if (ssd_scan_varlen_workspace_size(total_len, batch, nheads, head_dim, ngroups, dstate,
                                       chunk_size) == 0)
        return total_len < 0 || batch < 0 || nheads <= 0 || head_dim <= 0 || ngroups <= 0 ||
                       dstate <= 0 || chunk_size <= 0 || nheads % ngroups != 0
                   ? SSD_ERR_INVALID_ARG
                   : SSD_ERR_UNSUPPORTED;
    if (batch == 0)
        return SSD_OK;
    if (!A || !ssm_pool || max_slots < 0 || !cache_indices_host ||
        !qsl_valid(query_start_loc_host, total_len, batch))
        return SSD_ERR_INVALID_ARG;
    if (total_len > 0 && (!y_host || !x_host || !dt_host || !B_host || !C_host))
        return SSD_ERR_INVALID_ARG;
    for (int32_t b = 0; b < batch; ++b)
        if (static_cast<int64_t>(cache_indices_host[b]) >= max_slots)
            return SSD_ERR_INVALID_ARG;
    Plan pl;
    if (!make_plan(pl, query_start_loc_host, has_initial_state_host, cache_indices_host,
                   total_len, batch, nheads, head_dim, ngroups, dstate, chunk_size, pieces))
        return SSD_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < pl.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return SSD_ERR_WORKSPACE;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t HP = static_cast<size_t>(nheads) * head_dim;
    const size_t GN = static_cast<size_t>(ngroups) * dstate;
    const size_t rx = HP * 2, rdt = static_cast<size_t>(nheads) * 2, rb = GN * 2;  // bytes per token
    const uint8_t *hx = static_cast<const uint8_t *>(x_host);
    const uint8_t *hdt = static_cast<const uint8_t *>(dt_host);
    const uint8_t *hB = static_cast<const uint8_t *>(B_host);
    const uint8_t *hC = static_cast<const uint8_t *>(C_host);
    uint8_t *hy = static_cast<uint8_t *>(y_host);
    const ssd::StateIO io0{ssm_pool, nullptr, max_slots, nullptr, nullptr, 0};

    // every piece's host-side checks and tensor maps before anything is
    // queued, so that a host-side error status means nothing was copied,
    // launched or written
    for (const Piece &pc : pl.pieces) {
        const size_t a = static_cast<size_t>(pc.a), n = static_cast<size_t>(pc.e - pc.a);
        const size_t b = pc.cidx.size();
        uint8_t *m = ws + pc.meta_off;
        ssd::StateIO io = io0;
        io.cache_indices = reinterpret_cast<const uint32_t *>(m + (b + 1) * 4);
        const ssd_status_t st = ssd::scan_impl(
            ws + pl.y_off + a * rx, ws + pl.x_off + a * rx, ws + pl.dt_off + a * rdt, A,
            ws + pl.B_off + a * rb, ws + pl.C_off + a * rb, D, dt_bias, io,
            reinterpret_cast<const int32_t *>(m), m + (b + 1) * 4 + b * 4,
            static_cast<int64_t>(n), pc.batch(), nheads, head_dim, ngroups, dstate, chunk_size,
            dt_softplus, ws + pc.ws_off, pc.ws_bytes, stream_, nullptr, nullptr, false);
        if (st != SSD_OK)
            return st;
    }

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceStreams *ds = nullptr;
    if (device_streams(&ds) != cudaSuccess)
        return SSD_ERR_CUDA;
    const int np = static_cast<int>(pl.pieces.size());
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };

    // the directory and every piece's small arrays, written into a pinned
    // ring slot and copied with one copy ahead of the inputs
    const int slot = static_cast<int>(ds->next++ % kRing);
    if (ds->stage_used[slot] && !ok(cudaEventSynchronize(ds->stage_done[slot])))
        return SSD_ERR_CUDA;
    if (ds->stage_bytes[slot] < pl.meta_end) {
        if (ds->stage[slot] && !ok(cudaFreeHost(ds->stage[slot])))
            return SSD_ERR_CUDA;
        ds->stage[slot] = nullptr;
        ds->stage_bytes[slot] = 0;
        void *h = nullptr;
        if (!ok(cudaHostAlloc(&h, pl.meta_end, cudaHostAllocDefault)))
            return SSD_ERR_CUDA;
        ds->stage[slot] = static_cast<uint8_t *>(h);
        ds->stage_bytes[slot] = pl.meta_end;
    }
    uint8_t *hs = ds->stage[slot];
    Directory dir;
    std::memset(&dir, 0, sizeof dir);
    dir.magic = kDirMagic;
    dir.pieces = static_cast<uint32_t>(np);
    for (int k = 0; k < np; ++k)
        dir.scan_ws[k] = pl.pieces[k].ws_off;
    std::memcpy(hs, &dir, sizeof dir);
    for (const Piece &pc : pl.pieces) {
        const size_t b = pc.cidx.size();
        std::memcpy(hs + pc.meta_off, pc.qsl.data(), (b + 1) * 4);
        std::memcpy(hs + pc.meta_off + (b + 1) * 4, pc.cidx.data(), b * 4);
        std::memcpy(hs + pc.meta_off + (b + 1) * 4 + b * 4, pc.hinit.data(), b);
    }
    if (!ok(cudaEventRecord(ds->start, stream)) || !ok(cudaStreamWaitEvent(ds->h2d, ds->start, 0)) ||
        !ok(cudaStreamWaitEvent(ds->d2h, ds->start, 0)) ||
        !ok(cudaMemcpyAsync(ws, hs, pl.meta_end, cudaMemcpyHostToDevice, ds->h2d)) ||
        !ok(cudaEventRecord(ds->stage_done[slot], ds->h2d)))
        return SSD_ERR_CUDA;
    ds->stage_used[slot] = true;
    // after a failure past this point, later work on `stream` still waits
    // for every copy already queued on the internal streams
    auto fail = [&](ssd_status_t st) {
        if (cudaEventRecord(ds->in_done[0], ds->h2d) == cudaSuccess)
            (void)cudaStreamWaitEvent(stream, ds->in_done[0], 0);
        if (cudaEventRecord(ds->end, ds->d2h) == cudaSuccess)
            (void)cudaStreamWaitEvent(stream, ds->end, 0);
        return st;
    };

    // inputs, piece by piece, on the copy-in stream
    for (int k = 0; k < np; ++k) {
        const Piece &pc = pl.pieces[k];
        const size_t a = static_cast<size_t>(pc.a), n = static_cast<size_t>(pc.e - pc.a);
        if (n > 0 &&
            (!ok(cudaMemcpyAsync(ws + pl.x_off + a * rx, hx + a * rx, n * rx,
                                 cudaMemcpyHostToDevice, ds->h2d)) ||
             !ok(cudaMemcpyAsync(ws + pl.dt_off + a * rdt, hdt + a * rdt, n * rdt,
                                 cudaMemcpyHostToDevice, ds->h2d)) ||
             !ok(cudaMemcpyAsync(ws + pl.B_off + a * rb, hB + a * rb, n * rb,
                                 cudaMemcpyHostToDevice, ds->h2d)) ||
             !ok(cudaMemcpyAsync(ws + pl.C_off + a * rb, hC + a * rb, n * rb,
                                 cudaMemcpyHostToDevice, ds->h2d))))
            return fail(SSD_ERR_CUDA);
        if (!ok(cudaEventRecord(ds->in_done[k], ds->h2d)))
            return fail(SSD_ERR_CUDA);
    }

    // each piece's scan on the caller's stream once its inputs landed, and
    // its y back on the copy-out stream once the scan is done
    for (int k = 0; k < np; ++k) {
        const Piece &pc = pl.pieces[k];
        const size_t a = static_cast<size_t>(pc.a), n = static_cast<size_t>(pc.e - pc.a);
        const size_t b = pc.cidx.size();
        uint8_t *m = ws + pc.meta_off;
        ssd::StateIO io = io0;
        io.cache_indices = reinterpret_cast<const uint32_t *>(m + (b + 1) * 4);
        if (!ok(cudaStreamWaitEvent(stream, ds->in_done[k], 0)))
            return fail(SSD_ERR_CUDA);
        const ssd_status_t st = ssd::scan_impl(
            ws + pl.y_off + a * rx, ws + pl.x_off + a * rx, ws + pl.dt_off + a * rdt, A,
            ws + pl.B_off + a * rb, ws + pl.C_off + a * rb, D, dt_bias, io,
            reinterpret_cast<const int32_t *>(m), m + (b + 1) * 4 + b * 4,
            static_cast<int64_t>(n), pc.batch(), nheads, head_dim, ngroups, dstate, chunk_size,
            dt_softplus, ws + pc.ws_off, pc.ws_bytes, stream_, nullptr, nullptr);
        if (st != SSD_OK)
            return fail(st);
        if (!ok(cudaEventRecord(ds->scan_done[k], stream)) ||
            !ok(cudaStreamWaitEvent(ds->d2h, ds->scan_done[k], 0)))
            return fail(SSD_ERR_CUDA);
        if (n > 0 && !ok(cudaMemcpyAsync(hy + a * rx, ws + pl.y_off + a * rx, n * rx,
                                         cudaMemcpyDeviceToHost, ds->d2h)))
            return fail(SSD_ERR_CUDA);
    }
    if (!ok(cudaEventRecord(ds->end, ds->d2h)) || !ok(cudaStreamWaitEvent(stream, ds->end, 0)))
        return fail(SSD_ERR_CUDA);
    return SSD_OK;
}

ssd_status_t ssd_scan_varlen_host_read_errors(const void *workspace, ssd_stream_t stream_,
                                              uint32_t *flags)
{
    if (!workspace || !flags)
        return SSD_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    Directory dir;
    if (cudaMemcpyAsync(&dir, workspace, sizeof dir, cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (dir.magic != kDirMagic || dir.pieces == 0 || dir.pieces > kMaxPieces)
        return SSD_ERR_INVALID_ARG;
    uint32_t v = 0;
    for (uint32_t k = 0; k < dir.pieces; ++k) {
        uint32_t w = 0;
        const uint8_t *src = static_cast<const uint8_t *>(workspace) + dir.scan_ws[k];
        if (cudaMemcpyAsync(&w, src, sizeof w, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return SSD_ERR_CUDA;
        v |= w;
    }
    *flags = v;
    return v ? SSD_ERR_DEVICE : SSD_OK;
}

}  // extern "C"
