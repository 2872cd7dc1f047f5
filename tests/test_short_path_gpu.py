"""Sequences of at most 12 tokens take the per-token kernel; longer ones the
chunked kernels.  Both must match the oracle, the boundary (12 vs 13 tokens)
included, and a short sequence must give the same bits alone or in a batch."""
from __future__ import annotations

import dataclasses

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


# dstate need not be a power of two (any multiple of 16 up to 256): 48, 80 and
# 144 pad the lanes of a state row and leave tiles of 64, 32 and 16 rows
@pytest.mark.parametrize("P,N,G", [(64, 128, 1), (32, 256, 2), (128, 16, 1), (64, 48, 1),
                                   (32, 80, 2), (16, 144, 1)])
def test_lengths_around_the_threshold(P, N, G):
    lens = [0, 1, 2, 3, 5, 8, 9, 12, 13, 16, 130]
    w = W.make_workload("short_mix", lens, 4, P, G, N, 128, max_slots=12, seed=P + N,
                        has_init_p=0.6)
    y, pool, _, ws = run_cuda(w)
    import mamba_ssd_chunked_varlen_gb300 as pkg
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    y_ref, pool_ref = recurrence.run_workload(w)
    check_y(y_to_f64(y), y_ref, what=f"P={P} N={N}")
    check_slots(pool.cpu().numpy(), pool_ref, w.ssm_pool, w, what=f"P={P} N={N}")


def test_short_sequence_alone_equals_in_batch():
    w = W.make_workload("short_batch", [5, 40, 1, 12], 4, 64, 1, 64, 128, max_slots=6, seed=61,
                        has_init_p=1.0)
    y_all, pool_all, _, _ = run_cuda(w)
    for b in (0, 2, 3):   # the short ones
        t0, t1 = int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])
        wa = dataclasses.replace(
            w, x=w.x[t0:t1], dt=w.dt[t0:t1], B=w.B[t0:t1], C=w.C[t0:t1],
            query_start_loc=np.array([0, t1 - t0], dtype=np.int32),
            has_initial_state=w.has_initial_state[b:b + 1], cache_indices=w.cache_indices[b:b + 1])
        y1, pool1, _, _ = run_cuda(wa)
        assert torch.equal(y1.view(torch.int16), y_all[t0:t1].view(torch.int16)), f"seq {b}: y"
        s = int(w.cache_indices[b])
        assert torch.equal(pool1[s].view(torch.int32), pool_all[s].view(torch.int32)), f"seq {b}: state"
