"""The profiled entry point (ssd_scan_varlen_fwd_profiled) runs the same
kernels as ssd_scan_varlen_fwd with an event between the launches and no
programmatic overlap, so y and the pool must be bit-identical to the plain
call's, on a one-sequence call, a batch with short sequences, a call that uses
the block table and a call that takes the fused walk; the five events must be
recorded in stage order (non-negative elapsed times).
"""
from __future__ import annotations

import numpy as np
import pytest

from mamba_ssd_chunked_varlen_gb300 import workloads as W

from helpers import check_all_heads, run_cuda, to_device

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


def _cases():
    rng = np.random.default_rng(601)
    table_lens = [int(v) for v in rng.choice([5, 13, 64, 128, 129, 300, 1024], size=120)]
    return [
        ("one_seq", [2000], 8, 64, 1, 128, 256, 0.0),
        ("short_mix", [0, 3, 12, 13, 200, 1, 777, 9], 8, 64, 2, 128, 256, 0.7),
        ("table", table_lens, 8, 64, 2, 128, 256, 0.5),
        ("walk", [4096, 0, 5, 4200], 128, 64, 8, 128, 256, 0.75),
    ]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_profiled_matches_plain_call(case):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    name, lens, H, P, G, N, Q, init_p = case
    w = W.make_workload(f"prof_{name}", lens, H, P, G, N, Q, max_slots=len(lens) + 5,
                        seed=602 + len(lens), has_init_p=init_p)
    if name == "walk":
        assert pkg.ssd_scan_varlen_fused_walk(w.total_len, w.batch, w.nheads, w.head_dim,
                                              w.ngroups, w.dstate, w.chunk_size)
    y_ref, pool_ref, _, _ = run_cuda(w)
    d = to_device(w)
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = pkg.alloc_workspace(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups, w.dstate,
                             w.chunk_size)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    pkg.ssd_scan_varlen_fwd_profiled(y, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                     d["dt_bias"], d["ssm_pool"], d["query_start_loc"],
                                     d["has_initial_state"], d["cache_indices"],
                                     chunk_size=w.chunk_size, dt_softplus=w.dt_softplus,
                                     workspace=ws, events=events)
    torch.cuda.synchronize()
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(d["ssm_pool"].view(torch.int32), pool_ref.view(torch.int32))
    for a, b in zip(events[:-1], events[1:]):
        assert a.elapsed_time(b) >= 0.0
    if name in ("short_mix", "table"):
        check_all_heads(w, y, d["ssm_pool"], what=f"profiled {name}")
