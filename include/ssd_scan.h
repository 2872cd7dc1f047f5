/*
 * ssd_scan.h -- C ABI of the GB300 (sm_103a) Mamba-2 SSD varlen forward
 * prefill scan.
 *
 * The operation is the one defined in the "Per-token recurrence" section of
 * the Modular page "mamba2_ssd_scan" (Mojo module), for every head h, channel
 * p and group g = h / (nheads / ngroups):
 *
 *     dt_t     = softplus(dt[t,h] + dt_bias[h])     (plain dt + dt_bias when
 *                                                    dt_softplus == 0)
 *     dA_t     = exp(A[h] * dt_t)
 *     state_n  = state_n * dA_t + dt_t * B[t,g,n] * x[t,h,p]
 *     y[t,h,p] = sum_n C[t,g,n] * state_n + D[h] * x[t,h,p]
 *
 * The state starts at zero at every query_start_loc boundary, or at
 * ssm_pool[cache_indices[b]] when has_initial_state[b] is set, and the state
 * after the last token of sequence b is written back in place into
 * ssm_pool[cache_indices[b]] (page "Mamba2SSDChunkScanVarlenFwdInplace",
 * description and "Tensor shapes").  It is evaluated in the chunked SSD form
 * described on the kernelindex page "Mamba chunk scan with segsum": chunks of
 * chunk_size tokens aligned to each sequence start, an intra-chunk diagonal
 * block, per-chunk states, an inter-chunk state recurrence, and the
 * off-diagonal contribution.
 *
 * Conventions for every entry point:
 *   - all tensor pointers are DEVICE pointers to contiguous row-major data
 *     with the shapes listed at ssd_scan_varlen_fwd (ssd_scan_varlen_fwd_host
 *     takes its per-step tensors in host memory, as documented there); the
 *     caller owns them;
 *   - calls are asynchronous on `stream`; no entry point except the two
 *     read_errors functions synchronizes;
 *   - a status other than SSD_OK from a host-side check means that nothing
 *     was launched and no memory was written.
 */
#ifndef SSD_SCAN_H_
#define SSD_SCAN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

/* Same type as the CUDA runtime's cudaStream_t (NULL = legacy default stream). */
typedef struct CUstream_st *ssd_stream_t;

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,   /* NULL required pointer, bad size, misaligned pointer */
    SSD_ERR_UNSUPPORTED = 2,   /* valid but not supported here (head_dim, dstate, chunk_size) */
    SSD_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than ssd_scan_varlen_workspace_size */
    SSD_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed */
    SSD_ERR_DEVICE = 5,        /* ssd_scan_varlen_read_errors found a device-side error flag */
    SSD_ERR_TOO_LARGE = 6      /* ssd_scan_varlen_fwd_noalloc: the sizes need more scratch than
                                  its built-in buffer (SSD_NOALLOC_SCRATCH_BYTES) */
} ssd_status_t;

/* Device-side error flags (bit mask) written into the workspace by a call and
 * returned by ssd_scan_varlen_read_errors.  Device code never traps: on a bad
 * index or a wait that runs out it records the flag and skips the work. */
#define SSD_DEVERR_BAD_QUERY_START_LOC 0x1u /* qsl[0] != 0, decreasing, or qsl[batch] != total_len:
                                               nothing is computed or written */
#define SSD_DEVERR_BAD_CACHE_INDEX     0x2u /* cache_indices[b] >= max_slots: that slot access is
                                               skipped (state read as zero, not written back) */
#define SSD_DEVERR_TIMEOUT             0x4u /* an on-chip wait (TMA / tensor-core completion)
                                               exceeded its limit; outputs are incomplete */

/* Largest dstate supported (MAX_DSTATE in the "comptime values" section of
 * the Modular page "mamba2_ssd_scan"). */
#define SSD_MAX_DSTATE 256

/* Bytes of device scratch memory that ssd_scan_varlen_fwd needs for these
 * sizes (chunk table, per-chunk dt / cumulative log-decay, per-chunk states).
 * Returns 0 when the sizes are invalid or unsupported.  The bound holds for
 * every query_start_loc with these total_len and batch. */
SSD_API size_t ssd_scan_varlen_workspace_size(int64_t total_len, int32_t batch, int32_t nheads,
                                      int32_t head_dim, int32_t ngroups, int32_t dstate,
                                      int32_t chunk_size);

/* The varlen forward scan with in-place pool write-back.
 *
 *   y                 bf16  (total_len, nheads, head_dim)     out: every row written
 *   x                 bf16  (total_len, nheads, head_dim)
 *   dt                bf16  (total_len, nheads)
 *   A                 fp32  (nheads)
 *   B, C              bf16  (total_len, ngroups, dstate)
 *   D                 fp32  (nheads)   or NULL (read as 0)
 *   dt_bias           fp32  (nheads)   or NULL (read as 0)
 *   ssm_pool          fp32  (max_slots, nheads, head_dim, dstate)  in/out
 *   query_start_loc   int32 (batch + 1): sequence b is tokens [qsl[b], qsl[b+1])
 *   has_initial_state uint8 (batch)    or NULL (all false); nonzero = true
 *   cache_indices     uint32 (batch): pool slot of sequence b; slots must be distinct
 *   dt_softplus       nonzero: apply softplus to dt + dt_bias
 *   workspace         device scratch of at least ssd_scan_varlen_workspace_size bytes,
 *                     256-byte aligned; owned by the caller; contents need no
 *                     initialisation and are overwritten; one call at a time per workspace
 *
 * Only the pool slots named by cache_indices are written (each with the
 * final state of its sequence, also for a zero-length sequence); every other
 * pool byte is left unchanged.  Supported: head_dim in {16, 32, 64, 128},
 * 16 <= dstate <= 256 a multiple of 16, chunk_size in {64, 128, 256},
 * nheads % ngroups == 0.  x, B, C, y must be 16-byte aligned.  chunk_size
 * only changes rounding: chunks longer than 128 tokens are processed as
 * 128-token blocks with the state passed between them.
 * batch == 0 returns SSD_OK without launching.
 * Device-data preconditions (qsl monotone from 0 to total_len, slots in
 * range) are checked on the device; see SSD_DEVERR_*. */
SSD_API ssd_status_t ssd_scan_varlen_fwd(
    void *y, const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, const float *dt_bias, float *ssm_pool, const int32_t *query_start_loc,
    const uint8_t *has_initial_state, const uint32_t *cache_indices,
    int64_t total_len, int32_t batch, int32_t nheads, int32_t head_dim, int32_t ngroups,
    int32_t dstate, int64_t max_slots, int32_t chunk_size, int32_t dt_softplus,
    void *workspace, size_t workspace_bytes, ssd_stream_t stream);

/* ssd_scan_varlen_fwd with a bf16 slot pool: ssm_pool is bf16 (max_slots,
 * nheads, head_dim, dstate), the storage type the "Mamba2SSDChunkScanVarlenFwd
 * Inplace" tensor shapes allow besides fp32 ("storage dtype only; the scan
 * accumulates in fp32").  Initial states are widened to fp32 when read; final
 * states are rounded to bf16 (nearest even) when written.  Other arguments,
 * results and errors as ssd_scan_varlen_fwd. */
SSD_API ssd_status_t ssd_scan_varlen_fwd_bf16_pool(
    void *y, const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, const float *dt_bias, void *ssm_pool, const int32_t *query_start_loc,
    const uint8_t *has_initial_state, const uint32_t *cache_indices,
    int64_t total_len, int32_t batch, int32_t nheads, int32_t head_dim, int32_t ngroups,
    int32_t dstate, int64_t max_slots, int32_t chunk_size, int32_t dt_softplus,
    void *workspace, size_t workspace_bytes, ssd_stream_t stream);

/* Elements (not bytes) between consecutive tokens of each token-major input
 * and of y; 0 means contiguous (H*P for x and y, H for dt, G*N for B and C).
 * Within a token, x / y rows stay (H, P) contiguous, B / C rows (G, N) and dt
 * (H).  This is the layout of column slices of one wider buffer, e.g. x, B, C
 * and dt cut from a fused projection output (the per-tensor stride metadata
 * of the "mamba2_ssd_scan" comptime values Strides1D..Strides4D). */
typedef struct {
    int64_t x, dt, B, C, y;
} ssd_token_strides_t;

/* ssd_scan_varlen_fwd on strided token-major tensors.  Each nonzero stride
 * must be at least the contiguous one; the strides of x, B, C and y must be
 * multiples of 8 elements (16 bytes: TMA row pitch, 16-byte y stores), else
 * SSD_ERR_INVALID_ARG.  dt's stride is free.  strides == NULL is
 * ssd_scan_varlen_fwd.  Other arguments, results and errors as
 * ssd_scan_varlen_fwd. */
SSD_API ssd_status_t ssd_scan_varlen_fwd_strided(
    void *y, const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, const float *dt_bias, float *ssm_pool, const int32_t *query_start_loc,
    const uint8_t *has_initial_state, const uint32_t *cache_indices,
    int64_t total_len, int32_t batch, int32_t nheads, int32_t head_dim, int32_t ngroups,
    int32_t dstate, int64_t max_slots, int32_t chunk_size, int32_t dt_softplus,
    const ssd_token_strides_t *strides, void *workspace, size_t workspace_bytes,
    ssd_stream_t stream);

/* The same scan with separate state arrays instead of the slot pool: the form
 * of the "mamba2_ssd_scan" module description, whose state "resets to zero (or
 * to initial_states)" at each sequence start and whose final_states
 * (batch, nheads, head_dim, dstate) is "written at each sequence end"; the
 * in-place op of "Mamba2SSDChunkScanVarlenFwdInplace" differs only in reading
 * and writing these through ssm_pool[cache_indices[b]].
 *
 *   initial_states    fp32 (batch, nheads, head_dim, dstate) or NULL (zero
 *                     initial states); 16-byte aligned
 *   has_initial_state uint8 (batch) or NULL; when given, sequence b starts
 *                     from initial_states[b] only if has_initial_state[b] is
 *                     nonzero (zero otherwise); when NULL every sequence starts
 *                     from initial_states[b] (or zero if that is NULL)
 *   final_states      fp32 (batch, nheads, head_dim, dstate) out, 16-byte
 *                     aligned; row b written for every sequence, also of
 *                     length 0 (with its initial state); may alias
 *                     initial_states (each element is read before it is written)
 *
 * Every other argument, the workspace size, the supported sizes and the errors
 * are those of ssd_scan_varlen_fwd (NULL final_states with batch > 0:
 * SSD_ERR_INVALID_ARG). */
SSD_API ssd_status_t ssd_scan_varlen_fwd_states(
    void *y, const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, const float *dt_bias, const float *initial_states,
    const uint8_t *has_initial_state, float *final_states, const int32_t *query_start_loc,
    int64_t total_len, int32_t batch, int32_t nheads, int32_t head_dim, int32_t ngroups,
    int32_t dstate, int32_t chunk_size, int32_t dt_softplus, void *workspace,
    size_t workspace_bytes, ssd_stream_t stream);

/* ssd_scan_varlen_fwd with per-stage timing: `events` points to 5 CUDA events
 * (cudaEvent_t, created by the caller) that are recorded on `stream` before
 * the first stage and after each of the four stages (chunk state, state
 * passing, chunk scan, short sequences; a stage that does not run for these
 * sizes gets its two events back to back); cudaEventElapsedTime between
 * consecutive events gives each stage's device time.  Otherwise identical to
 * ssd_scan_varlen_fwd (same arguments, results and errors).  The records
 * separate the launches (no overlap between stages), so use it to attribute
 * time, not to time the whole call.  With batch == 0 nothing is launched and
 * no event is recorded. */
SSD_API ssd_status_t ssd_scan_varlen_fwd_profiled(
    void *y, const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, const float *dt_bias, float *ssm_pool, const int32_t *query_start_loc,
    const uint8_t *has_initial_state, const uint32_t *cache_indices,
    int64_t total_len, int32_t batch, int32_t nheads, int32_t head_dim, int32_t ngroups,
    int32_t dstate, int64_t max_slots, int32_t chunk_size, int32_t dt_softplus,
    void *workspace, size_t workspace_bytes, ssd_stream_t stream, void *const *events);

/* Size of the scratch buffer built into the library for
 * ssd_scan_varlen_fwd_noalloc (64 MiB of device memory on every GPU that
 * loads the library, held until the process exits). */
#define SSD_NOALLOC_SCRATCH_BYTES (64u << 20)

/* The scan for callers that cannot allocate device memory.  The pages have
 * no counterpart to this entry point; it exists for host code that may not
 * call cudaMalloc or any allocating library routine, such as a plugin inside
 * a host framework that owns all device memory and hands out no allocator,
 * or a serving loop that forbids allocation once it is running.
 *
 * Same arguments, results and errors as ssd_scan_varlen_fwd, minus the
 * workspace: the scratch lives in a fixed SSD_NOALLOC_SCRATCH_BYTES device
 * array inside the library.  Sizes whose ssd_scan_varlen_workspace_size
 * exceeds it return SSD_ERR_TOO_LARGE without launching (64 MiB fits, for
 * example, one 4096-token sequence with nheads 16, head_dim 64, dstate 256).  The caller still passes every input and output.
 *
 * Every call looks up the array's address on the current device
 * (cudaGetSymbolAddress, which allocates nothing); the first call on a device
 * may make CUDA load the library's device code there, so make that first call
 * before any stream capture.  It allocates nothing, now or later.  All calls on a device share the one
 * array and it keeps the last call's contents (each call rewrites everything
 * it reads, so nothing needs clearing); calls whose execution overlaps on the
 * GPU (different streams, or different host threads) race on it and must be
 * serialised by the caller.  Device-side error flags (SSD_DEVERR_*) of these
 * calls stay in the built-in array and are not reported. */
SSD_API ssd_status_t ssd_scan_varlen_fwd_noalloc(
    void *y, const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, const float *dt_bias, float *ssm_pool, const int32_t *query_start_loc,
    const uint8_t *has_initial_state, const uint32_t *cache_indices,
    int64_t total_len, int32_t batch, int32_t nheads, int32_t head_dim, int32_t ngroups,
    int32_t dstate, int64_t max_slots, int32_t chunk_size, int32_t dt_softplus,
    ssd_stream_t stream);

/* Synchronizes `stream` and returns the device-side error flags (SSD_DEVERR_*)
 * recorded by the last call that used `workspace`.  Returns SSD_ERR_DEVICE if
 * any flag is set, SSD_OK otherwise. */
SSD_API ssd_status_t ssd_scan_varlen_read_errors(const void *workspace, ssd_stream_t stream,
                                         uint32_t *flags);

/* ---- End-to-end call with host buffers --------------------------------
 *
 * The pages have no counterpart to this entry point.  It is for a caller
 * whose per-step tensors live in host memory: it copies them in, runs the
 * scan and copies y back, and overlaps the three.  The token range is cut
 * into up to SSD_HOST_MAX_PIECES pieces.  Piece k's inputs are copied on one
 * internal stream, its scan runs on `stream` once they have landed, and its
 * y is copied back on a second internal stream while later pieces are still
 * copied in or computed.
 *
 * Cuts fall on a sequence boundary or inside a sequence at a multiple of the
 * block length (min(chunk_size, 128) tokens) from its start, so every block
 * is the one the single call would form.  A sequence cut in two runs as two
 * parts: the first writes its running state to the sequence's slot, and the
 * second starts from that slot (as a continuation with an initial state).
 * The running state is fp32 in both cases, so the result matches one
 * ssd_scan_varlen_fwd call within the parity bounds.  The pieces' kernels
 * run one after another on `stream`.
 *
 * Arguments as ssd_scan_varlen_fwd, except:
 *   y_host, x_host, dt_host, B_host, C_host   host memory, same shapes and types;
 *                          pinned (page-locked) memory is needed for the overlap
 *                          (pageable memory works, but its copies do not overlap)
 *   query_start_loc_host, has_initial_state_host (or NULL), cache_indices_host
 *                          host arrays; checked on the host (qsl from 0, never
 *                          decreasing, ending at total_len; slots < max_slots):
 *                          SSD_ERR_INVALID_ARG without launching otherwise
 *   A, D, dt_bias, ssm_pool   device memory, as for ssd_scan_varlen_fwd
 *   pieces                 number of pieces asked for (0: one per ~6 MiB of
 *                          x, dt, B and C, 1 to SSD_HOST_MAX_PIECES); fewer
 *                          are used when cuts coincide
 *   workspace              device scratch of at least
 *                          ssd_scan_varlen_host_workspace_size bytes (256-byte
 *                          aligned).  It holds the device copies of the
 *                          inputs and of y and one scan workspace per piece.
 *
 * Host memory must stay valid until `stream` has passed the call (y_host is
 * written by then).  All work is ordered after earlier work on `stream`, and
 * later work on `stream` is ordered after all of it.  The two internal copy
 * streams of each device are created on the first call and are shared by
 * all calls on that device, so calls from several streams serialise their
 * copies.  The pieces' small arrays (local query_start_loc, slots, flags)
 * are written at call time into one of four pinned host buffers per device
 * that the library keeps (grown as needed, held until the process exits);
 * a call waits on the host only if that buffer's copy from four calls
 * earlier has not run yet.  So the call cannot be captured into a CUDA
 * graph.  Device-side error flags are read with
 * ssd_scan_varlen_host_read_errors.
 *
 * Every piece's host-side checks (and its tensor maps) run before the first
 * copy is queued, so a host-side error status means, as for the other entry
 * points, that nothing was copied, launched or written.  Only a failure of
 * the CUDA runtime itself after the first copy was queued (SSD_ERR_CUDA) can
 * leave earlier pieces launched: their y rows and slots are then written,
 * and a sequence cut between a launched and a failed piece holds its
 * mid-sequence state in its slot. */
#define SSD_HOST_MAX_PIECES 8

/* Bytes of workspace ssd_scan_varlen_fwd_host needs for this call (0 when
 * the sizes are unsupported or query_start_loc_host is invalid). */
SSD_API size_t ssd_scan_varlen_host_workspace_size(const int32_t *query_start_loc_host,
                                                   int64_t total_len, int32_t batch,
                                                   int32_t nheads, int32_t head_dim,
                                                   int32_t ngroups, int32_t dstate,
                                                   int32_t chunk_size, int32_t pieces);

/* The token positions where ssd_scan_varlen_fwd_host cuts this call: writes
 * the cuts (strictly increasing, inside (0, total_len)) to cuts_out, at most
 * SSD_HOST_MAX_PIECES - 1 of them, and returns the number of pieces (cuts +
 * 1), or -1 when query_start_loc_host is invalid or chunk_size unsupported.
 * Host only: no device call. */
SSD_API int32_t ssd_scan_varlen_host_plan(const int32_t *query_start_loc_host, int64_t total_len,
                                          int32_t batch, int32_t nheads, int32_t head_dim,
                                          int32_t ngroups, int32_t dstate, int32_t chunk_size,
                                          int32_t pieces, int64_t *cuts_out);

SSD_API ssd_status_t ssd_scan_varlen_fwd_host(
    void *y_host, const void *x_host, const void *dt_host, const float *A, const void *B_host,
    const void *C_host, const float *D, const float *dt_bias, float *ssm_pool,
    const int32_t *query_start_loc_host, const uint8_t *has_initial_state_host,
    const uint32_t *cache_indices_host, int64_t total_len, int32_t batch, int32_t nheads,
    int32_t head_dim, int32_t ngroups, int32_t dstate, int64_t max_slots, int32_t chunk_size,
    int32_t dt_softplus, int32_t pieces, void *workspace, size_t workspace_bytes,
    ssd_stream_t stream);

/* Synchronizes `stream` and returns the OR of the device-side error flags
 * (SSD_DEVERR_*) of every piece of the last ssd_scan_varlen_fwd_host call
 * that used `workspace`.  Returns SSD_ERR_DEVICE if any flag is set. */
SSD_API ssd_status_t ssd_scan_varlen_host_read_errors(const void *workspace, ssd_stream_t stream,
                                                      uint32_t *flags);

/* Test hook of the bounded-wait failure path (the pages have no counterpart).
 * With limit_ns > 0, every later call's chunk-state kernel (or fused scan
 * kernel) also waits, after its input copies have landed, on an on-chip
 * barrier that nothing completes; the wait gives up after limit_ns, the
 * kernel records SSD_DEVERR_TIMEOUT, frees its tensor memory and returns, as
 * it does when a real wait runs out (limit 1 s).  The outputs of such a call
 * are incomplete.  0 (the default) turns the hook off.  Process-wide; not
 * for production use. */
SSD_API void ssd_scan_varlen_test_stall(uint32_t limit_ns);

/* A static string naming a status code. */
SSD_API const char *ssd_status_string(ssd_status_t status);

/* Number of CUDA kernels one ssd_scan_varlen_fwd call launches for these sizes
 * (0 when batch == 0): chunk state and state passing (one fused kernel when
 * ssd_scan_varlen_fused_walk says so), chunk scan when total_len > 0, the
 * short-sequence kernel when the call may hold short sequences, and a
 * block-map kernel for batches of more than 512 sequences or calls whose
 * chunk-scan grid would run more than four waves of one CTA per SM.  Used to
 * count launches when timing.  Reads the current device's SM count and L2
 * size. */
SSD_API int32_t ssd_scan_varlen_num_launches(int64_t total_len, int32_t batch, int32_t nheads,
                                             int32_t head_dim, int32_t ngroups, int32_t dstate,
                                             int32_t chunk_size);

/* 1 when a call with these sizes computes the chunk states and the
 * inter-chunk state recurrence of the kernelindex page "Mamba chunk scan with
 * segsum" in one persistent kernel that keeps the chunk states on chip (calls
 * of long sequences -- 2048 tokens or more on average -- whose chunk states
 * would exceed the L2 and whose (sequence, head group) items fill the GPU), 0
 * when it writes them out and runs the recurrence as a kernel of its own.
 * Both compute the same result up to rounding; this only says which kernels
 * run.  0 for invalid sizes.  Reads the current device's SM count and L2
 * size (152 SMs, 126 MB when no device answers). */
SSD_API int32_t ssd_scan_varlen_fused_walk(int64_t total_len, int32_t batch, int32_t nheads,
                                           int32_t head_dim, int32_t ngroups, int32_t dstate,
                                           int32_t chunk_size);

/* The longest sequence (in tokens) that a call with these sizes gives to the
 * short-sequence kernel, the per-token recurrence of the Modular page
 * "mamba2_ssd_scan" ("Per-token recurrence"), instead of the chunked kernels:
 * 12 when the call holds several sequences or total_len <= 12, else 0.  Both
 * paths compute the same recurrence; this only says which kernel runs. */
SSD_API int32_t ssd_scan_varlen_short_threshold(int64_t total_len, int32_t batch);

#ifdef __cplusplus
}
#endif

#endif /* SSD_SCAN_H_ */
