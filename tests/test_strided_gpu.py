"""Strided token-major inputs (ssd_scan_varlen_fwd_strided): x, B, C and dt as
column slices of one fused projection output and y as a slice of a wider
buffer.  The arithmetic is that of the contiguous call, so the results must be
bit-identical to it, and within tolerance of the oracle."""
from __future__ import annotations

import numpy as np
import pytest

from mamba_ssd_chunked_varlen_gb300 import workloads as W
from oracle import recurrence

from helpers import check_slots, check_y, run_cuda, to_device, y_to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mamba_ssd_chunked_varlen_gb300 as pkg
    from mamba_ssd_chunked_varlen_gb300 import build
    build.build()
    pkg.library()


def _fused_views(w, d, pad):
    """One (T, width) bf16 buffer holding [pad | x | pad | B | C | dt | pad] per token;
    returns views x, B, C, dt into it (column offsets multiples of 8 elements)."""
    T, H, P, G, N = w.total_len, w.nheads, w.head_dim, w.ngroups, w.dstate
    o_x = pad
    o_b = o_x + H * P + pad
    o_c = o_b + G * N
    o_dt = o_c + G * N
    width = o_dt + H + pad + (-(o_dt + H + pad)) % 8
    buf = torch.full((T, width), float("nan"), dtype=torch.bfloat16, device="cuda")
    buf[:, o_x:o_x + H * P] = d["x"].reshape(T, H * P)
    buf[:, o_b:o_b + G * N] = d["B"].reshape(T, G * N)
    buf[:, o_c:o_c + G * N] = d["C"].reshape(T, G * N)
    buf[:, o_dt:o_dt + H] = d["dt"]
    x = buf[:, o_x:o_x + H * P].unflatten(1, (H, P))
    B = buf[:, o_b:o_b + G * N].unflatten(1, (G, N))
    C = buf[:, o_c:o_c + G * N].unflatten(1, (G, N))
    dt = buf[:, o_dt:o_dt + H]
    return x, B, C, dt, width


@pytest.mark.parametrize("name,pad", [("kernelindex", 8), ("ragged", 16), ("small", 24)])
def test_strided_matches_contiguous_and_oracle(name, pad):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    if name == "small":
        w = W.make_workload("strided_small", [300, 1, 129, 0, 64], 6, 32, 2, 64, 64, max_slots=7,
                            seed=91, has_init_p=0.5)
    else:
        w = W.workload(name)
    y_ref_gpu, pool_ref_gpu, _, _ = run_cuda(w)
    d = to_device(w)
    x, B, C, dt, width = _fused_views(w, d, pad)
    T, H, P = w.total_len, w.nheads, w.head_dim
    ywide = torch.full((T, H * P + 2 * pad), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = ywide[:, pad:pad + H * P].unflatten(1, (H, P))
    ws = pkg.alloc_workspace(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups, w.dstate,
                             w.chunk_size)
    pkg.ssd_scan_varlen_fwd_strided(y, x, dt, d["A"], B, C, d["D"], d["dt_bias"], d["ssm_pool"],
                                    d["query_start_loc"], d["has_initial_state"],
                                    d["cache_indices"], chunk_size=w.chunk_size,
                                    dt_softplus=w.dt_softplus, workspace=ws)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    # bit-identical to the contiguous call
    assert torch.equal(y.contiguous().view(torch.int16), y_ref_gpu.view(torch.int16))
    assert torch.equal(d["ssm_pool"].view(torch.int32), pool_ref_gpu.view(torch.int32))
    # the padding columns of y are untouched
    assert torch.isnan(ywide[:, :pad].float()).all() and torch.isnan(ywide[:, pad + H * P:].float()).all()
    # and within tolerance of the oracle
    y_ref, pool_ref = recurrence.run_workload(w)
    check_y(y_to_f64(y), y_ref, what=f"strided {name}")
    check_slots(d["ssm_pool"].cpu().numpy(), pool_ref, w.ssm_pool, w, what=f"strided {name}")


def test_strided_rejects_unaligned_pitch():
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.workload("tiny")
    d = to_device(w)
    T, H, P = w.total_len, w.nheads, w.head_dim
    buf = torch.zeros((T, H * P + 4), dtype=torch.bfloat16, device="cuda")   # pitch % 8 != 0
    x = buf[:, :H * P].unflatten(1, (H, P))
    y = torch.empty((T, H, P), dtype=torch.bfloat16, device="cuda")
    ws = pkg.alloc_workspace(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups, w.dstate,
                             w.chunk_size)
    with pytest.raises(pkg.SSDError) as e:
        pkg.ssd_scan_varlen_fwd_strided(y, x, d["dt"], d["A"], d["B"], d["C"], d["D"],
                                        d["dt_bias"], d["ssm_pool"], d["query_start_loc"],
                                        d["has_initial_state"], d["cache_indices"],
                                        chunk_size=w.chunk_size, workspace=ws)
    assert e.value.status == 1
