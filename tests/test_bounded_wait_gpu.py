"""The bounded-wait failure path of the kernels, driven on the GPU without a
fault: the test hook ssd_scan_varlen_test_stall makes the chunk-state kernel
wait, after its input copies have landed, on an on-chip barrier that nothing
completes.  The wait must give up after the given limit, the call must
return (the stream drains), SSD_DEVERR_TIMEOUT must be reported through the
workspace, and the context must stay usable: the next call without the hook
matches the oracle.
"""
from __future__ import annotations

import time

import pytest

from mamba_ssd_chunked_varlen_gb300 import workloads as W
from oracle import recurrence

from helpers import check_slots, check_y, run_cuda, y_to_f64

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


def test_a_wait_that_runs_out_sets_the_timeout_flag_and_returns(pkg):
    w = W.make_workload("stall", [300], 4, 64, 1, 64, 128, max_slots=2, seed=90,
                        has_init_p=1.0)
    limit_ns = 2_000_000   # 2 ms instead of the kernels' 1 s
    pkg.ssd_scan_varlen_test_stall(limit_ns)
    try:
        t0 = time.perf_counter()
        _, _, _, ws = run_cuda(w)
        flags = pkg.ssd_scan_varlen_read_errors(ws)   # synchronizes: the kernels returned
        elapsed = time.perf_counter() - t0
    finally:
        pkg.ssd_scan_varlen_test_stall(0)
    assert flags & pkg.binding.DEVERR_TIMEOUT, f"flags {flags:#x}"
    assert not flags & (pkg.binding.DEVERR_BAD_QUERY_START_LOC | pkg.binding.DEVERR_BAD_CACHE_INDEX)
    assert elapsed < 30.0
    # the context is still usable and the hook is off again
    y, pool, _, ws2 = run_cuda(w)
    assert pkg.ssd_scan_varlen_read_errors(ws2) == 0
    y_ref, pool_ref = recurrence.run_workload(w)
    check_y(y_to_f64(y), y_ref, what="after the stalled call")
    check_slots(pool.cpu().numpy(), pool_ref, w.ssm_pool, w, what="after the stalled call")
