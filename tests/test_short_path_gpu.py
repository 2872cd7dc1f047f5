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


def _sub_run(w, lo, hi, pool):
    """Sequences [lo, hi) of `w` as a call of their own on `pool`."""
    t0, t1 = int(w.query_start_loc[lo]), int(w.query_start_loc[hi])
    return dataclasses.replace(
        w, x=w.x[t0:t1], dt=w.dt[t0:t1], B=w.B[t0:t1], C=w.C[t0:t1],
        query_start_loc=(w.query_start_loc[lo:hi + 1] - t0).astype(np.int32),
        has_initial_state=w.has_initial_state[lo:hi], cache_indices=w.cache_indices[lo:hi],
        ssm_pool=pool)


def test_large_batch_block_table():
    """More than 512 sequences: a block-map kernel writes a block table that the
    block kernels read.  Every sequence must give the bits it gives in a call
    small enough for each CTA to map its own block (no block-map kernel), and
    the whole must match the oracle."""
    rng = np.random.default_rng(71)
    lens = rng.choice([0, 1, 3, 7, 12, 13, 40, 128, 129, 300], size=700)
    w = W.make_workload("big_batch", [int(v) for v in lens], 4, 32, 2, 32, 64,
                        max_slots=720, seed=72, has_init_p=0.6)
    import mamba_ssd_chunked_varlen_gb300 as pkg
    assert pkg.ssd_scan_varlen_num_launches(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups,
                                            w.dstate, w.chunk_size) == 5
    y, pool, _, ws = run_cuda(w)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    y_ref, pool_ref = recurrence.run_workload(w)
    check_y(y_to_f64(y), y_ref, what="700 sequences")
    check_slots(pool.cpu().numpy(), pool_ref, w.ssm_pool, w, what="700 sequences")
    # the same sequences in calls of 35, each mapping its blocks per CTA
    pool_k = w.ssm_pool
    for lo in range(0, w.batch, 35):
        hi = min(w.batch, lo + 35)
        wk = _sub_run(w, lo, hi, pool_k)
        assert pkg.ssd_scan_varlen_num_launches(wk.total_len, wk.batch, wk.nheads, wk.head_dim,
                                                wk.ngroups, wk.dstate, wk.chunk_size) == 4
        yk, poolk, _, _ = run_cuda(wk)
        t0, t1 = int(w.query_start_loc[lo]), int(w.query_start_loc[hi])
        assert torch.equal(y[t0:t1].view(torch.int16), yk.view(torch.int16)), f"sequences [{lo}, {hi})"
        pool_k = poolk.cpu().numpy()
    assert np.array_equal(pool.cpu().numpy().view(np.int32), pool_k.view(np.int32))


def test_large_batch_bad_query_start_loc():
    import mamba_ssd_chunked_varlen_gb300 as pkg
    from helpers import to_device
    w = W.make_workload("big_bad", [5] * 600, 2, 32, 1, 32, 64, max_slots=600, seed=73)
    d = to_device(w)
    qsl = w.query_start_loc.copy()
    qsl[300] = qsl[301] + 1          # a negative length
    d["query_start_loc"] = torch.from_numpy(qsl).cuda()
    pool_before = d["ssm_pool"].clone()
    y, pool, _, ws = run_cuda(w, dev=d)
    flags = pkg.ssd_scan_varlen_read_errors(ws)
    assert flags & pkg.binding.DEVERR_BAD_QUERY_START_LOC
    assert not flags & pkg.binding.DEVERR_TIMEOUT
    assert torch.equal(pool_before, pool)
    assert torch.isnan(y.float()).all()
