"""Python binding of the C ABI in include/ssd_scan.h (ctypes).

Argument marshalling only: every step of the scan runs in the CUDA kernels of
libssd_scan.so.  Tensors are torch CUDA tensors (torch provides device memory
and streams); their shapes give the sizes passed to the C ABI.  There is no
CPU fallback: if the library is not built, or a tensor is not on a CUDA
device, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libssd_scan.so")

# Every symbol include/ssd_scan.h declares.
EXPORTED_SYMBOLS = (
    "ssd_scan_varlen_workspace_size",
    "ssd_scan_varlen_fwd",
    "ssd_scan_varlen_fwd_profiled",
    "ssd_scan_varlen_fwd_states",
    "ssd_scan_varlen_fwd_strided",
    "ssd_scan_varlen_fwd_bf16_pool",
    "ssd_scan_varlen_fwd_noalloc",
    "ssd_scan_varlen_read_errors",
    "ssd_status_string",
    "ssd_scan_varlen_num_launches",
    "ssd_scan_varlen_fused_walk",
    "ssd_scan_varlen_short_threshold",
    "ssd_scan_varlen_host_workspace_size",
    "ssd_scan_varlen_host_plan",
    "ssd_scan_varlen_fwd_host",
    "ssd_scan_varlen_host_read_errors",
    "ssd_scan_varlen_test_stall",
)

HOST_MAX_PIECES = 8  # SSD_HOST_MAX_PIECES

SSD_OK = 0
SSD_ERR_TOO_LARGE = 6
NOALLOC_SCRATCH_BYTES = 64 << 20  # SSD_NOALLOC_SCRATCH_BYTES
DEVERR_BAD_QUERY_START_LOC = 0x1
DEVERR_BAD_CACHE_INDEX = 0x2
DEVERR_TIMEOUT = 0x4

_lib: Optional[ctypes.CDLL] = None


class TokenStrides(ctypes.Structure):
    """ssd_token_strides_t: elements between consecutive tokens (0: contiguous)."""
    _fields_ = [("x", ctypes.c_int64), ("dt", ctypes.c_int64), ("B", ctypes.c_int64),
                ("C", ctypes.c_int64), ("y", ctypes.c_int64)]


class SSDError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


def library() -> ctypes.CDLL:
    """Load libssd_scan.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "mamba_ssd_chunked_varlen_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.ssd_scan_varlen_workspace_size.restype = sz
    lib.ssd_scan_varlen_workspace_size.argtypes = [i64, i32, i32, i32, i32, i32, i32]
    lib.ssd_scan_varlen_fwd.restype = ctypes.c_int
    lib.ssd_scan_varlen_fwd.argtypes = ([vp] * 12 + [i64, i32, i32, i32, i32, i32, i64, i32, i32]
                                        + [vp, sz, vp])
    lib.ssd_scan_varlen_fwd_profiled.restype = ctypes.c_int
    lib.ssd_scan_varlen_fwd_profiled.argtypes = lib.ssd_scan_varlen_fwd.argtypes + [vp]
    lib.ssd_scan_varlen_fwd_states.restype = ctypes.c_int
    lib.ssd_scan_varlen_fwd_states.argtypes = ([vp] * 12 + [i64, i32, i32, i32, i32, i32, i32, i32]
                                               + [vp, sz, vp])
    lib.ssd_scan_varlen_fwd_strided.restype = ctypes.c_int
    lib.ssd_scan_varlen_fwd_strided.argtypes = (lib.ssd_scan_varlen_fwd.argtypes[:21]
                                                + [ctypes.POINTER(TokenStrides), vp, sz, vp])
    lib.ssd_scan_varlen_fwd_bf16_pool.restype = ctypes.c_int
    lib.ssd_scan_varlen_fwd_bf16_pool.argtypes = lib.ssd_scan_varlen_fwd.argtypes
    lib.ssd_scan_varlen_fwd_noalloc.restype = ctypes.c_int
    lib.ssd_scan_varlen_fwd_noalloc.argtypes = lib.ssd_scan_varlen_fwd.argtypes[:21] + [vp]
    lib.ssd_scan_varlen_read_errors.restype = ctypes.c_int
    lib.ssd_scan_varlen_read_errors.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_status_string.argtypes = [ctypes.c_int]
    lib.ssd_scan_varlen_num_launches.restype = i32
    lib.ssd_scan_varlen_num_launches.argtypes = [i64, i32, i32, i32, i32, i32, i32]
    lib.ssd_scan_varlen_fused_walk.restype = i32
    lib.ssd_scan_varlen_fused_walk.argtypes = [i64, i32, i32, i32, i32, i32, i32]
    lib.ssd_scan_varlen_short_threshold.restype = i32
    lib.ssd_scan_varlen_short_threshold.argtypes = [i64, i32]
    lib.ssd_scan_varlen_host_workspace_size.restype = sz
    lib.ssd_scan_varlen_host_workspace_size.argtypes = [vp, i64, i32, i32, i32, i32, i32, i32, i32]
    lib.ssd_scan_varlen_host_plan.restype = i32
    lib.ssd_scan_varlen_host_plan.argtypes = [vp, i64, i32, i32, i32, i32, i32, i32, i32,
                                              ctypes.POINTER(ctypes.c_int64)]
    lib.ssd_scan_varlen_fwd_host.restype = ctypes.c_int
    lib.ssd_scan_varlen_fwd_host.argtypes = ([vp] * 12 + [i64, i32, i32, i32, i32, i32, i64, i32,
                                                          i32, i32] + [vp, sz, vp])
    lib.ssd_scan_varlen_test_stall.restype = None
    lib.ssd_scan_varlen_test_stall.argtypes = [ctypes.c_uint32]
    lib.ssd_scan_varlen_host_read_errors.restype = ctypes.c_int
    lib.ssd_scan_varlen_host_read_errors.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return library().ssd_status_string(int(status)).decode()


def ssd_scan_varlen_workspace_size(total_len: int, batch: int, nheads: int, head_dim: int,
                                   ngroups: int, dstate: int, chunk_size: int) -> int:
    return int(library().ssd_scan_varlen_workspace_size(total_len, batch, nheads, head_dim,
                                                        ngroups, dstate, chunk_size))


def ssd_scan_varlen_num_launches(total_len: int, batch: int, nheads: int, head_dim: int,
                                 ngroups: int, dstate: int, chunk_size: int) -> int:
    return int(library().ssd_scan_varlen_num_launches(total_len, batch, nheads, head_dim,
                                                      ngroups, dstate, chunk_size))


def ssd_scan_varlen_fused_walk(total_len: int, batch: int, nheads: int, head_dim: int,
                               ngroups: int, dstate: int, chunk_size: int) -> bool:
    """True when a call of these sizes runs the fused chunk-state walk (one
    kernel for the chunk states and the state recurrence) instead of the two
    split kernels."""
    return bool(library().ssd_scan_varlen_fused_walk(total_len, batch, nheads, head_dim,
                                                     ngroups, dstate, chunk_size))


def ssd_scan_varlen_short_threshold(total_len: int, batch: int) -> int:
    return int(library().ssd_scan_varlen_short_threshold(total_len, batch))


def _ptr(t, what: str, dtype=None, allow_none: bool = False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{what} is required")
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must have dtype {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() > 0 else ctypes.c_void_p(t.data_ptr() or 0)


def _stream_handle(stream) -> ctypes.c_void_p:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _fwd_args(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc, has_initial_state,
              cache_indices, chunk_size, dt_softplus, workspace, stream, pool_dtype=None):
    import torch
    pool_dtype = torch.float32 if pool_dtype is None else pool_dtype
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    batch = query_start_loc.shape[0] - 1
    if workspace is None:
        raise ValueError("workspace is required (see ssd_scan_varlen_workspace_size)")
    if has_initial_state is not None and has_initial_state.dtype == torch.bool:
        has_initial_state = has_initial_state.view(torch.uint8)
    if cache_indices.dtype not in (torch.int32, torch.uint32):
        raise ValueError("cache_indices must be int32 or uint32")
    return (
        _ptr(y, "y", torch.bfloat16), _ptr(x, "x", torch.bfloat16),
        _ptr(dt, "dt", torch.bfloat16), _ptr(A, "A", torch.float32),
        _ptr(B, "B", torch.bfloat16), _ptr(C, "C", torch.bfloat16),
        _ptr(D, "D", torch.float32, True), _ptr(dt_bias, "dt_bias", torch.float32, True),
        _ptr(ssm_pool, "ssm_pool", pool_dtype), _ptr(query_start_loc, "query_start_loc",
                                                     torch.int32),
        _ptr(has_initial_state, "has_initial_state", torch.uint8, True),
        _ptr(cache_indices, "cache_indices"),
        T, batch, H, P, G, N, ssm_pool.shape[0], int(chunk_size), int(bool(dt_softplus)),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream_handle(stream))


def ssd_scan_varlen_fwd_profiled(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc,
                                 has_initial_state, cache_indices, *, chunk_size: int,
                                 dt_softplus: bool = True, workspace=None, stream=None,
                                 events=None) -> None:
    """ssd_scan_varlen_fwd that also records 5 torch.cuda.Event objects around
    the four stages (chunk state, state passing, chunk scan, short sequences)."""
    if events is None or len(events) != 5:
        raise ValueError("events must be 5 torch.cuda.Event objects")
    import torch
    for e in events:
        if e.cuda_event == 0:  # torch creates the CUDA event lazily, on first record
            e.record(torch.cuda.current_stream() if stream is None else stream)
    handles = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    st = library().ssd_scan_varlen_fwd_profiled(
        *_fwd_args(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc, has_initial_state,
                   cache_indices, chunk_size, dt_softplus, workspace, stream), handles)
    if st != SSD_OK:
        raise SSDError(st, "ssd_scan_varlen_fwd_profiled")


def ssd_scan_varlen_fwd(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc,
                        has_initial_state, cache_indices, *, chunk_size: int,
                        dt_softplus: bool = True, workspace=None, stream=None) -> None:
    """Run the scan on `stream` (default: torch's current stream).

    Shapes: y, x (T, H, P) bf16; dt (T, H) bf16; A (H,) fp32; B, C (T, G, N)
    bf16; D, dt_bias (H,) fp32 or None; ssm_pool (slots, H, P, N) fp32 (updated
    in place); query_start_loc (batch+1,) int32; has_initial_state (batch,)
    uint8/bool or None; cache_indices (batch,) int32/uint32 (same bits);
    workspace: a uint8 CUDA tensor of at least ssd_scan_varlen_workspace_size
    bytes.
    """
    st = library().ssd_scan_varlen_fwd(
        *_fwd_args(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc, has_initial_state,
                   cache_indices, chunk_size, dt_softplus, workspace, stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_scan_varlen_fwd")


def ssd_scan_varlen_fwd_states(y, x, dt, A, B, C, D, dt_bias, initial_states,
                               has_initial_state, final_states, query_start_loc, *,
                               chunk_size: int, dt_softplus: bool = True, workspace=None,
                               stream=None) -> None:
    """The scan with separate state arrays instead of the slot pool:
    initial_states (batch, H, P, N) fp32 or None (zero initial states),
    has_initial_state (batch,) uint8/bool or None (None: every sequence starts
    from initial_states), final_states (batch, H, P, N) fp32 written for every
    sequence.  Other arguments as ssd_scan_varlen_fwd."""
    import torch
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    batch = query_start_loc.shape[0] - 1
    if workspace is None:
        raise ValueError("workspace is required (see ssd_scan_varlen_workspace_size)")
    if has_initial_state is not None and has_initial_state.dtype == torch.bool:
        has_initial_state = has_initial_state.view(torch.uint8)
    for name, t in (("initial_states", initial_states), ("final_states", final_states)):
        if t is not None and tuple(t.shape) != (batch, H, P, N):
            raise ValueError(f"{name} must have shape {(batch, H, P, N)}")
    st = library().ssd_scan_varlen_fwd_states(
        _ptr(y, "y", torch.bfloat16), _ptr(x, "x", torch.bfloat16),
        _ptr(dt, "dt", torch.bfloat16), _ptr(A, "A", torch.float32),
        _ptr(B, "B", torch.bfloat16), _ptr(C, "C", torch.bfloat16),
        _ptr(D, "D", torch.float32, True), _ptr(dt_bias, "dt_bias", torch.float32, True),
        _ptr(initial_states, "initial_states", torch.float32, True),
        _ptr(has_initial_state, "has_initial_state", torch.uint8, True),
        _ptr(final_states, "final_states", torch.float32),
        _ptr(query_start_loc, "query_start_loc", torch.int32),
        T, batch, H, P, G, N, int(chunk_size), int(bool(dt_softplus)),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream_handle(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_scan_varlen_fwd_states")


def _token_major(t, what: str, dtype, inner: int):
    """Pointer and token stride of a token-major view whose rows (the trailing
    `inner` elements) are contiguous."""
    if t is None:
        raise ValueError(f"{what} is required")
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{what} must have dtype {dtype}, got {t.dtype}")
    if t.dim() < 2 or t[0].numel() != inner or (t.shape[0] > 0 and not t[0].is_contiguous()):
        raise ValueError(f"{what}: each token's row must be contiguous")
    return ctypes.c_void_p(t.data_ptr()), t.stride(0)


def ssd_scan_varlen_fwd_strided(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc,
                                has_initial_state, cache_indices, *, chunk_size: int,
                                dt_softplus: bool = True, workspace=None, stream=None) -> None:
    """ssd_scan_varlen_fwd on token-major views with any token stride (e.g.
    x, B, C, dt as column slices of a fused projection output, y a slice of a
    wider buffer); each token's row must be contiguous."""
    import torch
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    batch = query_start_loc.shape[0] - 1
    if workspace is None:
        raise ValueError("workspace is required (see ssd_scan_varlen_workspace_size)")
    if has_initial_state is not None and has_initial_state.dtype == torch.bool:
        has_initial_state = has_initial_state.view(torch.uint8)
    py, sy = _token_major(y, "y", torch.bfloat16, H * P)
    px, sx = _token_major(x, "x", torch.bfloat16, H * P)
    pdt, sdt = _token_major(dt, "dt", torch.bfloat16, H)
    pb, sb = _token_major(B, "B", torch.bfloat16, G * N)
    pc, sc = _token_major(C, "C", torch.bfloat16, G * N)
    strides = TokenStrides(sx, sdt, sb, sc, sy)
    st = library().ssd_scan_varlen_fwd_strided(
        py, px, pdt, _ptr(A, "A", torch.float32), pb, pc, _ptr(D, "D", torch.float32, True),
        _ptr(dt_bias, "dt_bias", torch.float32, True), _ptr(ssm_pool, "ssm_pool", torch.float32),
        _ptr(query_start_loc, "query_start_loc", torch.int32),
        _ptr(has_initial_state, "has_initial_state", torch.uint8, True),
        _ptr(cache_indices, "cache_indices"), T, batch, H, P, G, N, ssm_pool.shape[0],
        int(chunk_size), int(bool(dt_softplus)), ctypes.byref(strides),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream_handle(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_scan_varlen_fwd_strided")


def ssd_scan_varlen_fwd_bf16_pool(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc,
                                  has_initial_state, cache_indices, *, chunk_size: int,
                                  dt_softplus: bool = True, workspace=None, stream=None) -> None:
    """ssd_scan_varlen_fwd with a bf16 ssm_pool (slots, H, P, N): initial states
    widened to fp32 on read, final states rounded to bf16 on write."""
    import torch
    st = library().ssd_scan_varlen_fwd_bf16_pool(
        *_fwd_args(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc, has_initial_state,
                   cache_indices, chunk_size, dt_softplus, workspace, stream,
                   pool_dtype=torch.bfloat16))
    if st != SSD_OK:
        raise SSDError(st, "ssd_scan_varlen_fwd_bf16_pool")


def ssd_scan_varlen_fwd_noalloc(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc,
                                has_initial_state, cache_indices, *, chunk_size: int,
                                dt_softplus: bool = True, stream=None) -> None:
    """The scan for callers that cannot allocate device memory: same as
    ssd_scan_varlen_fwd without a workspace; the scratch is the library's
    built-in NOALLOC_SCRATCH_BYTES array (sizes needing more raise SSDError
    with status SSD_ERR_TOO_LARGE).  Calls that overlap on the GPU race on
    that array; serialise them."""
    import torch
    args = _fwd_args(y, x, dt, A, B, C, D, dt_bias, ssm_pool, query_start_loc,
                     has_initial_state, cache_indices, chunk_size, dt_softplus,
                     torch.empty(0, dtype=torch.uint8, device=x.device), stream)
    st = library().ssd_scan_varlen_fwd_noalloc(*args[:21], args[23])
    if st != SSD_OK:
        raise SSDError(st, "ssd_scan_varlen_fwd_noalloc")


def ssd_scan_varlen_read_errors(workspace, stream=None) -> int:
    """Synchronize the stream and return the device-side error flags."""
    import torch
    flags = ctypes.c_uint32(0)
    st = library().ssd_scan_varlen_read_errors(_ptr(workspace, "workspace", torch.uint8),
                                               _stream_handle(stream), ctypes.byref(flags))
    if st not in (SSD_OK, 5):
        raise SSDError(st, "ssd_scan_varlen_read_errors")
    return int(flags.value)


def ssd_scan_varlen_test_stall(limit_ns: int) -> None:
    """Test hook: later calls wait on a never-completed on-chip barrier that
    gives up after `limit_ns` (0 turns the hook off)."""
    library().ssd_scan_varlen_test_stall(int(limit_ns))


def alloc_workspace(total_len: int, batch: int, nheads: int, head_dim: int, ngroups: int,
                    dstate: int, chunk_size: int, device="cuda"):
    """A uint8 torch tensor of the size the C ABI asks for."""
    import torch
    n = ssd_scan_varlen_workspace_size(total_len, batch, nheads, head_dim, ngroups, dstate,
                                       chunk_size)
    if n == 0:
        raise SSDError(2, "ssd_scan_varlen_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


# ---- end-to-end call with host buffers

def _hptr(t, what: str, dtype=None, allow_none: bool = False):
    """Pointer to a contiguous CPU tensor (pinned for overlapped copies)."""
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{what} is required")
    if t.is_cuda:
        raise ValueError(f"{what} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must have dtype {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr() or 0)


def _host_qsl(query_start_loc_host):
    import torch
    if query_start_loc_host.is_cuda or query_start_loc_host.dtype != torch.int32:
        raise ValueError("query_start_loc_host must be an int32 CPU tensor")
    return query_start_loc_host.contiguous()


def ssd_scan_varlen_host_plan(query_start_loc_host, nheads: int, head_dim: int, ngroups: int,
                              dstate: int, chunk_size: int, pieces: int = 0):
    """Token positions where ssd_scan_varlen_fwd_host cuts a call (a list of
    cuts; pieces = len + 1).  Host only."""
    q = _host_qsl(query_start_loc_host)
    batch = q.numel() - 1
    total = int(q[-1]) if batch >= 0 else 0
    out = (ctypes.c_int64 * HOST_MAX_PIECES)()
    n = library().ssd_scan_varlen_host_plan(ctypes.c_void_p(q.data_ptr()), total, batch,
                                            nheads, head_dim, ngroups, dstate,
                                            int(chunk_size), int(pieces), out)
    if n < 0:
        raise SSDError(1, "ssd_scan_varlen_host_plan")
    return [int(out[i]) for i in range(n - 1)]


def ssd_scan_varlen_host_workspace_size(query_start_loc_host, nheads: int, head_dim: int,
                                        ngroups: int, dstate: int, chunk_size: int,
                                        pieces: int = 0) -> int:
    q = _host_qsl(query_start_loc_host)
    batch = q.numel() - 1
    return int(library().ssd_scan_varlen_host_workspace_size(
        ctypes.c_void_p(q.data_ptr()), int(q[-1]), batch, nheads, head_dim, ngroups, dstate,
        int(chunk_size), int(pieces)))


def alloc_host_workspace(query_start_loc_host, nheads: int, head_dim: int, ngroups: int,
                         dstate: int, chunk_size: int, pieces: int = 0, device="cuda"):
    import torch
    n = ssd_scan_varlen_host_workspace_size(query_start_loc_host, nheads, head_dim, ngroups,
                                            dstate, chunk_size, pieces)
    if n == 0:
        raise SSDError(2, "ssd_scan_varlen_host_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def ssd_scan_varlen_fwd_host(y_host, x_host, dt_host, A, B_host, C_host, D, dt_bias, ssm_pool,
                             query_start_loc_host, has_initial_state_host, cache_indices_host,
                             *, chunk_size: int, dt_softplus: bool = True, pieces: int = 0,
                             workspace=None, stream=None) -> None:
    """The scan with y, x, dt, B, C and the int arrays in host memory (CPU
    tensors; pin them for overlapped copies) and A, D, dt_bias, ssm_pool on
    the device.  The inputs are copied in, scanned and y copied back in
    pieces that overlap; y_host is written once `stream` has passed the call.
    workspace: a uint8 CUDA tensor of ssd_scan_varlen_host_workspace_size
    bytes."""
    import torch
    if workspace is None:
        raise ValueError("workspace is required (see ssd_scan_varlen_host_workspace_size)")
    T, H, P = x_host.shape
    G, N = B_host.shape[1], B_host.shape[2]
    q = _host_qsl(query_start_loc_host)
    batch = q.numel() - 1
    if has_initial_state_host is not None and has_initial_state_host.dtype == torch.bool:
        has_initial_state_host = has_initial_state_host.view(torch.uint8)
    if cache_indices_host.dtype not in (torch.int32, torch.uint32):
        raise ValueError("cache_indices_host must be int32 or uint32")
    st = library().ssd_scan_varlen_fwd_host(
        _hptr(y_host, "y_host", torch.bfloat16), _hptr(x_host, "x_host", torch.bfloat16),
        _hptr(dt_host, "dt_host", torch.bfloat16), _ptr(A, "A", torch.float32),
        _hptr(B_host, "B_host", torch.bfloat16), _hptr(C_host, "C_host", torch.bfloat16),
        _ptr(D, "D", torch.float32, True), _ptr(dt_bias, "dt_bias", torch.float32, True),
        _ptr(ssm_pool, "ssm_pool", torch.float32), ctypes.c_void_p(q.data_ptr()),
        _hptr(has_initial_state_host, "has_initial_state_host", torch.uint8, True),
        _hptr(cache_indices_host, "cache_indices_host"),
        T, batch, H, P, G, N, ssm_pool.shape[0], int(chunk_size), int(bool(dt_softplus)),
        int(pieces), _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
        _stream_handle(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_scan_varlen_fwd_host")


def ssd_scan_varlen_host_read_errors(workspace, stream=None) -> int:
    """Synchronize the stream and return the OR of the device-side error flags
    of the last ssd_scan_varlen_fwd_host call that used this workspace."""
    import torch
    flags = ctypes.c_uint32(0)
    st = library().ssd_scan_varlen_host_read_errors(_ptr(workspace, "workspace", torch.uint8),
                                                    _stream_handle(stream), ctypes.byref(flags))
    if st not in (SSD_OK, 5):
        raise SSDError(st, "ssd_scan_varlen_host_read_errors")
    return int(flags.value)
