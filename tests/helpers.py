"""Shared helpers of the GPU tests: move a workload to the device, run the CUDA
path through the C ABI, and compare with the oracle at the stated tolerances.

Tolerances (the target accuracy of this op):
  y      per element |y - y_ref| <= 1e-2 * max|y_ref| + 1 bf16 ulp of y_ref
  state  per written slot  ||S - S_ref||_2 / ||S_ref||_2 <= 1e-3
  routing (query_start_loc / cache_indices handling) bit-exact; untouched
  slots byte-identical.
"""
from __future__ import annotations

import numpy as np

Y_REL = 1e-2
STATE_REL_L2 = 1e-3


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (bf16 keeps 8 of fp32's 24 significant bits)."""
    a = np.abs(np.asarray(v, dtype=np.float64)).astype(np.float32)
    return np.spacing(a).astype(np.float64) * 65536.0


def to_device(w, device="cuda"):
    import torch

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)

    def f32(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)

    return dict(
        x=bf(w.x), dt=bf(w.dt), A=f32(w.A), B=bf(w.B), C=bf(w.C), D=f32(w.D),
        dt_bias=f32(w.dt_bias), ssm_pool=f32(w.ssm_pool),
        query_start_loc=torch.from_numpy(np.ascontiguousarray(w.query_start_loc, np.int32)).to(device),
        has_initial_state=(None if w.has_initial_state is None else
                           torch.from_numpy(np.ascontiguousarray(w.has_initial_state, np.uint8)).to(device)),
        cache_indices=torch.from_numpy(w.cache_indices.astype(np.int64).astype(np.int32)).to(device),
    )


def run_cuda(w, chunk_size=None, dev=None, workspace=None, stream=None):
    """Run the CUDA path on workload `w`.  Returns (y bf16 tensor, pool tensor,
    device inputs, workspace)."""
    import torch
    import mamba_ssd_chunked_varlen_gb300 as pkg
    Q = w.chunk_size if chunk_size is None else chunk_size
    d = to_device(w) if dev is None else dev
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    if workspace is None:
        workspace = pkg.alloc_workspace(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups,
                                        w.dstate, Q)
    pkg.ssd_scan_varlen_fwd(y, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"],
                            d["ssm_pool"], d["query_start_loc"], d["has_initial_state"],
                            d["cache_indices"], chunk_size=Q, dt_softplus=w.dt_softplus,
                            workspace=workspace, stream=stream)
    return y, d["ssm_pool"], d, workspace


def y_to_f64(y) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def check_y(y_gpu: np.ndarray, y_ref: np.ndarray, rows=None, what=""):
    """Element-wise bound; `rows` selects token rows (default: all)."""
    if rows is not None:
        y_gpu, y_ref = y_gpu[rows], y_ref[rows]
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite output"
    if y_ref.size == 0:
        return 0.0
    bound = Y_REL * np.abs(y_ref).max() + bf16_ulp(y_ref)
    err = np.abs(y_gpu - y_ref)
    worst = float((err / bound).max())
    assert worst <= 1.0, (f"{what}: y outside tolerance, max |d| = {err.max():.3e}, "
                          f"max |y_ref| = {np.abs(y_ref).max():.3e}, worst ratio {worst:.3f}")
    return worst


def check_slots(pool_gpu: np.ndarray, pool_ref: np.ndarray, pool_in: np.ndarray, w,
                heads=None, seqs=None, what=""):
    """Written slots within relative L2; every other slot byte-identical to the input."""
    written = {}
    for b, s in enumerate(w.cache_indices):
        if seqs is None or b in seqs:
            written[int(s)] = b
    worst = 0.0
    hs = slice(None) if heads is None else slice(*heads)
    for s in written:
        ref = pool_ref[s][hs].astype(np.float64)
        got = pool_gpu[s][hs].astype(np.float64)
        nrm = np.linalg.norm(ref)
        rel = np.linalg.norm(got - ref) / nrm if nrm > 0 else np.linalg.norm(got)
        worst = max(worst, rel)
        assert rel <= STATE_REL_L2, f"{what}: slot {s} relative L2 {rel:.3e}"
    all_written = set(int(s) for s in w.cache_indices)
    for s in range(pool_in.shape[0]):
        if s not in all_written:
            assert np.array_equal(pool_gpu[s].view(np.uint32), pool_in[s].view(np.uint32)), \
                f"{what}: untouched slot {s} changed"
    return worst


def check_all_heads(w, y, pool, what="", span=16):
    """Every head of every sequence against one full oracle run: y at the y
    tolerance, written slots at the state tolerance, untouched slots
    byte-identical.  The comparison runs over head ranges of at most `span`
    heads at a time, each inside one B/C group when the group size allows,
    which bounds the host memory of the temporaries on the largest
    workloads."""
    from oracle import recurrence
    y_ref, pool_ref = recurrence.run_workload(w)
    yg = y_to_f64(y) if hasattr(y, "cpu") else y
    pg = pool.cpu().numpy() if hasattr(pool, "cpu") else pool
    hpg = w.nheads // w.ngroups
    step = hpg
    while step > span and step % 2 == 0:
        step //= 2
    worst_y = worst_s = 0.0
    for h0 in range(0, w.nheads, step):
        h1 = min(w.nheads, h0 + step)
        worst_y = max(worst_y, check_y(yg[:, h0:h1], y_ref[:, h0:h1],
                                       what=f"{what} heads ({h0}, {h1})"))
        worst_s = max(worst_s, check_slots(pg, pool_ref, w.ssm_pool, w, heads=(h0, h1),
                                           what=f"{what} heads ({h0}, {h1})"))
    return worst_y, worst_s

