"""Parity of the separate-state-array form (ssd_scan_varlen_fwd_states) with the
oracle.

The "mamba2_ssd_scan" form starts each sequence from initial_states[b] (or
zero) and writes final_states[b]; the in-place op of
"Mamba2SSDChunkScanVarlenFwdInplace" is the same computation with those rows
living in ssm_pool[cache_indices[b]].  So the expected values are the oracle's
in-place results with initial_states taken from the workload's pool rows:
y is the oracle's y and final_states[b] the oracle's pool slot cache_indices[b].
"""
from __future__ import annotations

import copy

import numpy as np
import pytest

from mamba_ssd_chunked_varlen_gb300 import workloads as W
from oracle import recurrence

from helpers import STATE_REL_L2, check_y, to_device, y_to_f64

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


def _run_states(w, init, flags, alias=False):
    """Run the states form; returns (y, final_states, initial_states after the call)."""
    import mamba_ssd_chunked_varlen_gb300 as pkg
    d = to_device(w)
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    shape = (w.batch, w.nheads, w.head_dim, w.dstate)
    init_t = None if init is None else torch.from_numpy(np.ascontiguousarray(init, np.float32)).cuda()
    flags_t = None if flags is None else torch.from_numpy(np.ascontiguousarray(flags, np.uint8)).cuda()
    if alias:
        final = init_t
    else:
        final = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    ws = pkg.alloc_workspace(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups, w.dstate,
                             w.chunk_size)
    pkg.ssd_scan_varlen_fwd_states(y, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                   d["dt_bias"], init_t, flags_t, final, d["query_start_loc"],
                                   chunk_size=w.chunk_size, dt_softplus=w.dt_softplus,
                                   workspace=ws)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    return (y_to_f64(y), final.cpu().numpy(),
            None if init_t is None or alias else init_t.cpu().numpy())


def _expect(w, effective_flags):
    """The oracle on the in-place form: pool slot cache_indices[b] = initial_states[b]."""
    wr = copy.copy(w)
    wr.has_initial_state = np.asarray(effective_flags, dtype=np.uint8)
    y_ref, pool_ref = recurrence.run_workload(wr)
    return y_ref, pool_ref[np.asarray(w.cache_indices, dtype=np.int64)]


def _check_final(final, final_ref, what):
    assert np.all(np.isfinite(final)), f"{what}: final_states not fully written"
    for b in range(final.shape[0]):
        ref = final_ref[b].astype(np.float64)
        nrm = np.linalg.norm(ref)
        rel = np.linalg.norm(final[b] - ref) / nrm if nrm > 0 else np.linalg.norm(final[b])
        assert rel <= STATE_REL_L2, f"{what}: final_states[{b}] relative L2 {rel:.3e}"


def _cases():
    ragged = W.workload("ragged")
    small = W.make_workload("states_small", [300, 1, 129, 64], 6, 32, 2, 64, 64, max_slots=6,
                            seed=77, has_init_p=0.5)
    short = W.make_workload("states_short", [0, 5, 0, 200, 1], 4, 64, 1, 128, 128, max_slots=7,
                            seed=78, has_init_p=0.5)
    return {"ragged": ragged, "small": small, "short": short}


@pytest.mark.parametrize("name", ["ragged", "small", "short"])
def test_states_form_with_flags(name):
    w = _cases()[name]
    init = w.ssm_pool[np.asarray(w.cache_indices, dtype=np.int64)]
    y, final, init_after = _run_states(w, init, w.has_initial_state)
    y_ref, final_ref = _expect(w, w.has_initial_state)
    check_y(y, y_ref, what=name)
    _check_final(final, final_ref, name)
    assert np.array_equal(init_after.view(np.uint32), init.astype(np.float32).view(np.uint32)), \
        f"{name}: initial_states changed"


def test_states_form_without_flags_uses_every_initial_state():
    w = _cases()["small"]
    init = w.ssm_pool[np.asarray(w.cache_indices, dtype=np.int64)]
    y, final, _ = _run_states(w, init, None)
    y_ref, final_ref = _expect(w, np.ones(w.batch, np.uint8))
    check_y(y, y_ref, what="no flags")
    _check_final(final, final_ref, "no flags")


def test_states_form_without_initial_states_starts_from_zero():
    w = _cases()["short"]
    y, final, _ = _run_states(w, None, np.ones(w.batch, np.uint8))
    y_ref, final_ref = _expect(w, np.zeros(w.batch, np.uint8))
    check_y(y, y_ref, what="no initial states")
    _check_final(final, final_ref, "no initial states")


def test_states_form_final_may_alias_initial():
    w = _cases()["ragged"]
    init = w.ssm_pool[np.asarray(w.cache_indices, dtype=np.int64)]
    y, final, _ = _run_states(w, init, w.has_initial_state, alias=True)
    y_ref, final_ref = _expect(w, w.has_initial_state)
    check_y(y, y_ref, what="aliased")
    _check_final(final, final_ref, "aliased")


def test_states_form_matches_in_place_bit_for_bit():
    """Same arithmetic, different addresses: y and the states agree exactly."""
    from helpers import run_cuda
    w = _cases()["ragged"]
    y_ip, pool, _, _ = run_cuda(w)
    init = w.ssm_pool[np.asarray(w.cache_indices, dtype=np.int64)]
    y, final, _ = _run_states(w, init, w.has_initial_state)
    assert np.array_equal(y_to_f64(y_ip), y)
    got = pool.cpu().numpy()[np.asarray(w.cache_indices, dtype=np.int64)]
    assert np.array_equal(got.view(np.uint32), final.view(np.uint32))
