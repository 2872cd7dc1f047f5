"""The no-allocation entry point, ssd_scan_varlen_fwd_noalloc.

Some callers of this library cannot allocate device memory: a plugin running
inside a host framework that owns all device memory and offers no allocator,
or a serving loop that forbids allocation once it is running.  For them the
library carries a fixed scratch array and this entry point takes no
workspace.  Here it is checked, through the C ABI, against the entry point
that takes a caller-allocated workspace, on two calls in a row with different problems (the second
call must not see anything of the first one's leftovers in the shared
array): y and the pool must be bit-identical to the workspace call's, which
runs the same launches, and within the tolerances of every other GPU test.  The file name makes pytest collect it last.
"""
from __future__ import annotations

import numpy as np
import pytest

from mamba_ssd_chunked_varlen_gb300 import workloads as W

from helpers import check_y, to_device, STATE_REL_L2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_varlen_gb300 import build
    build.build()
    import mamba_ssd_chunked_varlen_gb300 as p
    p.library()
    return p


def _run(pkg, w, noalloc: bool):
    d = to_device(w)
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    args = (y, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"], d["ssm_pool"],
            d["query_start_loc"], d["has_initial_state"], d["cache_indices"])
    if noalloc:
        pkg.ssd_scan_varlen_fwd_noalloc(*args, chunk_size=w.chunk_size,
                                        dt_softplus=w.dt_softplus)
    else:
        ws = pkg.alloc_workspace(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups,
                                 w.dstate, w.chunk_size)
        pkg.ssd_scan_varlen_fwd(*args, chunk_size=w.chunk_size, dt_softplus=w.dt_softplus,
                                workspace=ws)
        assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    torch.cuda.synchronize()
    return y.view(torch.int16).cpu().numpy(), d["ssm_pool"].cpu().numpy()


def _compare(w, got, ref):
    """The no-allocation call runs the same launches on the same sizes as the
    workspace call, so y (as bf16 bit patterns) and every pool slot must be
    bit-identical to the workspace call's; the tolerance check against it is
    kept as well, so that a mismatch reports how far apart the two are."""
    (y_n, pool_n), (y_r, pool_r) = got, ref
    y_nf = W.bf16_bits_to_f32(y_n.view(np.uint16)).astype(np.float64)
    y_rf = W.bf16_bits_to_f32(y_r.view(np.uint16)).astype(np.float64)
    check_y(y_nf, y_rf, what=f"{w.name} no-alloc vs workspace entry point")
    for s in set(int(v) for v in w.cache_indices):
        nrm = np.linalg.norm(pool_r[s])
        assert np.linalg.norm(pool_n[s] - pool_r[s]) <= STATE_REL_L2 * nrm
    np.testing.assert_array_equal(y_n, y_r)
    np.testing.assert_array_equal(pool_n.view(np.uint32), pool_r.view(np.uint32))
    untouched = set(range(w.max_slots)) - set(int(v) for v in w.cache_indices)
    for s in untouched:
        assert np.array_equal(pool_n[s].view(np.uint32), w.ssm_pool[s].view(np.uint32))


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row(pkg):
    first = W.workload("kernelindex")
    second = W.make_workload("noalloc2", [700, 1, 0, 333, 129], 8, 64, 2, 128, 128,
                             max_slots=9, seed=77, has_init_p=0.6)
    for w in (first, second):
        need = pkg.ssd_scan_varlen_workspace_size(w.total_len, w.batch, w.nheads, w.head_dim,
                                                  w.ngroups, w.dstate, w.chunk_size)
        assert 0 < need <= pkg.binding.NOALLOC_SCRATCH_BYTES
    ref1 = _run(pkg, first, noalloc=False)
    ref2 = _run(pkg, second, noalloc=False)
    got1 = _run(pkg, first, noalloc=True)
    got2 = _run(pkg, second, noalloc=True)
    _compare(first, got1, ref1)
    _compare(second, got2, ref2)


def test_noalloc_rejects_sizes_beyond_its_scratch(pkg):
    w = W.make_workload("big", [4200, 4200, 4200, 4200], 16, 64, 1, 256, 256, max_slots=4, seed=5)
    need = pkg.ssd_scan_varlen_workspace_size(w.total_len, w.batch, w.nheads, w.head_dim,
                                              w.ngroups, w.dstate, w.chunk_size)
    assert need > pkg.binding.NOALLOC_SCRATCH_BYTES
    with pytest.raises(pkg.SSDError) as e:
        _run(pkg, w, noalloc=True)
    assert e.value.status == pkg.binding.SSD_ERR_TOO_LARGE
