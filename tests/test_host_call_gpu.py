"""The host-buffer entry point (ssd_scan_varlen_fwd_host): inputs in pinned
host memory, copied in, scanned and y copied back piece by piece.

A single sequence cut on block boundaries runs exactly the blocks of one
device call, and the running state crosses each cut in fp32 through the
slot, so y and the slot must be bit-identical to ssd_scan_varlen_fwd.  Varlen
batches are cut inside sequences too (a continuation of 8 tokens takes the
short-sequence kernel, empty sequences sit at a cut and at the end); they are
compared with the oracle (fp64 per-token recurrence) at the parity
tolerances, untouched slots byte-identical.  Host-side argument checks
return an error without touching the pool.
"""
from __future__ import annotations

import numpy as np
import pytest

from mamba_ssd_chunked_varlen_gb300 import workloads as W
from oracle import recurrence

from helpers import check_slots, check_y, run_cuda, y_to_f64

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


def _host(w):
    """Pinned host tensors of the per-step inputs, device tensors of the rest."""
    as_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16))).view(
        torch.bfloat16).pin_memory()
    h = {"x": as_bf16(w.x), "dt": as_bf16(w.dt), "B": as_bf16(w.B), "C": as_bf16(w.C),
         "qsl": torch.from_numpy(w.query_start_loc.astype(np.int32)),
         "hinit": (None if w.has_initial_state is None else
                   torch.from_numpy(w.has_initial_state.astype(np.uint8))),
         "cidx": torch.from_numpy(w.cache_indices.astype(np.int64).astype(np.int32))}
    f32 = lambda a: None if a is None else torch.from_numpy(
        np.ascontiguousarray(a, np.float32)).cuda()
    d = {"A": f32(w.A), "D": f32(w.D), "dt_bias": f32(w.dt_bias), "pool": f32(w.ssm_pool)}
    return h, d


def _run_host(w, pieces, ws=None):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    h, d = _host(w)
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    if ws is None:
        ws = pkg.alloc_host_workspace(h["qsl"], w.nheads, w.head_dim, w.ngroups, w.dstate,
                                      w.chunk_size, pieces)
    pkg.ssd_scan_varlen_fwd_host(y, h["x"], h["dt"], d["A"], h["B"], h["C"], d["D"],
                                 d["dt_bias"], d["pool"], h["qsl"], h["hinit"], h["cidx"],
                                 chunk_size=w.chunk_size, dt_softplus=w.dt_softplus,
                                 pieces=pieces, workspace=ws)
    assert pkg.ssd_scan_varlen_host_read_errors(ws) == 0
    torch.cuda.synchronize()
    return y, d["pool"], h, ws


@pytest.mark.parametrize("pieces", [1, 2, 3, 0])
def test_single_sequence_bit_identical(pieces):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.make_workload("host_ki", [4096], 16, 64, 1, 256, 256, max_slots=4, seed=501,
                        has_init_p=1.0)
    n = len(pkg.ssd_scan_varlen_host_plan(torch.from_numpy(w.query_start_loc.astype(np.int32)),
                                          16, 64, 1, 256, w.chunk_size, pieces)) + 1
    assert n == (pieces if pieces > 0 else 2)   # 12.7 MB of inputs: two ~6 MiB pieces
    y_dev, pool_dev, _, _ = run_cuda(w)
    y_host, pool_host, _, _ = _run_host(w, pieces)
    assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
    assert torch.equal(pool_host.cpu(), pool_dev.cpu())
    y_ref, pool_ref = recurrence.run_workload(w, heads=(0, 2))
    check_y(y_to_f64(y_host)[:, 0:2], y_ref[:, 0:2], what=f"{pieces} pieces")
    check_slots(pool_host.cpu().numpy(), pool_ref, w.ssm_pool, w, heads=(0, 2))


@pytest.mark.parametrize("lens,Q,pieces,cuts", [
    # a one-block first part and an 8-token continuation (short-sequence
    # kernel), an empty sequence inside a piece and one at the end
    ([700, 136, 0, 900, 12, 600, 0], 128, 3, [828, 1604]),
    # 64-token chunks, five pieces
    ([700, 136, 0, 900, 12, 600, 0], 64, 5, [448, 964, 1412, 1876]),
    # an empty sequence right at the start of a piece
    ([520, 8, 0, 1100, 300], 128, 2, [912]),
])
def test_varlen_against_oracle(lens, Q, pieces, cuts):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.make_workload(f"host_varlen_{Q}_{pieces}", lens, 4, 32, 2, 64, Q, max_slots=12,
                        seed=502 + pieces, has_init_p=0.5)
    qsl = torch.from_numpy(w.query_start_loc.astype(np.int32))
    assert pkg.ssd_scan_varlen_host_plan(qsl, 4, 32, 2, 64, Q, pieces) == cuts
    y_host, pool_host, _, ws = _run_host(w, pieces)
    y_ref, pool_ref = recurrence.run_workload(w)
    check_y(y_to_f64(y_host), y_ref, what=f"{pieces} pieces")
    check_slots(pool_host.cpu().numpy(), pool_ref, w.ssm_pool, w)
    # the same workspace again: the same result
    y2, pool2, _, _ = _run_host(w, pieces, ws=ws)
    assert torch.equal(y2.view(torch.int16), y_host.view(torch.int16))
    assert torch.equal(pool2.cpu(), pool_host.cpu())


def test_host_checks_reject_before_launch():
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.make_workload("host_bad", [300, 200], 4, 32, 2, 64, 128, max_slots=4, seed=510,
                        has_init_p=1.0)
    h, d = _host(w)
    ws = pkg.alloc_host_workspace(h["qsl"], w.nheads, w.head_dim, w.ngroups, w.dstate, 128, 2)
    y = torch.zeros(w.x.shape, dtype=torch.bfloat16).pin_memory()
    before = d["pool"].clone()

    def call(qsl, cidx):
        pkg.ssd_scan_varlen_fwd_host(y, h["x"], h["dt"], d["A"], h["B"], h["C"], d["D"],
                                     d["dt_bias"], d["pool"], qsl, h["hinit"], cidx,
                                     chunk_size=128, pieces=2, workspace=ws)

    bad_qsl = h["qsl"].clone()
    bad_qsl[1] = 600          # decreasing
    with pytest.raises(pkg.SSDError) as e:
        call(bad_qsl, h["cidx"])
    assert e.value.status == 1
    bad_cidx = h["cidx"].clone()
    bad_cidx[0] = w.ssm_pool.shape[0]   # out of range
    with pytest.raises(pkg.SSDError) as e:
        call(h["qsl"], bad_cidx)
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert torch.equal(d["pool"], before)
    assert not y.view(torch.int16).any()


def test_back_to_back_calls_share_streams_and_ring():
    """Six calls queued without a sync in between, alternating two workloads
    and two workspaces: the library's shared copy streams, events and its
    four-slot pinned ring (wrapped once here) must keep every call's inputs
    and outputs apart.  Each result equals a device call on the same
    inputs."""
    import mamba_ssd_chunked_varlen_gb300 as pkg
    ws_all = [W.make_workload("host_b2b_a", [700, 136, 0, 900], 4, 32, 2, 64, 128,
                              max_slots=8, seed=520, has_init_p=0.5),
              W.make_workload("host_b2b_b", [2048, 40, 1500], 4, 32, 2, 64, 128,
                              max_slots=8, seed=521, has_init_p=0.5)]
    refs = []
    for w in ws_all:
        y_dev, pool_dev, _, _ = run_cuda(w)
        refs.append((y_dev.cpu(), pool_dev.cpu()))
    staged = []
    for w in ws_all:
        h, _ = _host(w)
        ws = pkg.alloc_host_workspace(h["qsl"], w.nheads, w.head_dim, w.ngroups, w.dstate,
                                      w.chunk_size, 3)
        staged.append((w, h, ws))
    # every call's device arguments (a fresh pool each) and pinned y made up
    # front, so that nothing between the calls waits for the device
    args = []
    for call in range(6):
        w = staged[call % 2][0]
        args.append((_host(w)[1],
                     torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16).pin_memory()))
    torch.cuda.synchronize()
    outs = []
    for call in range(6):
        w, h, ws = staged[call % 2]
        d, y = args[call]
        pkg.ssd_scan_varlen_fwd_host(y, h["x"], h["dt"], d["A"], h["B"], h["C"], d["D"],
                                     d["dt_bias"], d["pool"], h["qsl"], h["hinit"], h["cidx"],
                                     chunk_size=w.chunk_size, dt_softplus=w.dt_softplus,
                                     pieces=3, workspace=ws)
        outs.append((call % 2, y, d["pool"]))
    torch.cuda.synchronize()
    for k, y, pool in outs:
        y_ref, pool_ref = refs[k]
        # the pieces cut sequences, so the rounding differs slightly from one call
        check_y(y_to_f64(y), y_to_f64(y_ref), what=f"call of workload {k}")
        assert torch.allclose(pool.cpu(), pool_ref, rtol=1e-4, atol=1e-5)
    for _, _, ws in staged:
        assert pkg.ssd_scan_varlen_host_read_errors(ws) == 0


@pytest.mark.parametrize("pinned", [True, False])
def test_empty_optionals_and_pageable_memory(pinned):
    """D, dt_bias and has_initial_state absent (read as 0 / false), softplus
    off, and (pinned=False) inputs and y in pageable host memory: the copies
    then do not overlap, but the result is the same."""
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.make_workload("host_opt", [900, 0, 300, 7, 1200], 4, 32, 2, 64, 128, max_slots=8,
                        seed=530, with_D=False, with_dt_bias=False, dt_softplus=False)
    # no initial states in the workload: passing None for the flags means the same
    assert w.D is None and w.dt_bias is None and not w.has_initial_state.any()
    h, d = _host(w)
    if not pinned:
        h = {k: (v.clone() if v is not None else None) for k, v in h.items()}   # pageable
        assert not h["x"].is_pinned()
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16)
    if pinned:
        y = y.pin_memory()
    ws = pkg.alloc_host_workspace(h["qsl"], w.nheads, w.head_dim, w.ngroups, w.dstate,
                                  w.chunk_size, 3)
    pkg.ssd_scan_varlen_fwd_host(y, h["x"], h["dt"], d["A"], h["B"], h["C"], None, None,
                                 d["pool"], h["qsl"], None, h["cidx"], chunk_size=w.chunk_size,
                                 dt_softplus=False, pieces=3, workspace=ws)
    assert pkg.ssd_scan_varlen_host_read_errors(ws) == 0
    torch.cuda.synchronize()
    y_ref, pool_ref = recurrence.run_workload(w)
    check_y(y_to_f64(y), y_ref, what=f"pinned={pinned}")
    check_slots(d["pool"].cpu().numpy(), pool_ref, w.ssm_pool, w)
