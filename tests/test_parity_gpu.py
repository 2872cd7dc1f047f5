"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every test here needs a GPU.  Inputs are the seeded synthetic workloads of
mamba_ssd_chunked_varlen_gb300.workloads; expected values come from the oracle
(fp64 per-token recurrence) on the same inputs.
"""
from __future__ import annotations

import numpy as np
import pytest

from mamba_ssd_chunked_varlen_gb300 import workloads as W
from oracle import recurrence

from helpers import check_all_heads, check_slots, check_y, run_cuda, to_device, y_to_f64

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


def _check_full(w, chunk_size=None, what=""):
    y, pool, _, ws = run_cuda(w, chunk_size)
    import mamba_ssd_chunked_varlen_gb300 as pkg
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    y_ref, pool_ref = recurrence.run_workload(w)
    wy = check_y(y_to_f64(y), y_ref, what=what)
    ws_ = check_slots(pool.cpu().numpy(), pool_ref, w.ssm_pool, w, what=what)
    return wy, ws_


@pytest.mark.parametrize("name", ["tiny", "kernelindex", "ragged", "serving_mix"])
def test_workload_parity_full(name):
    w = W.workload(name)
    _check_full(w, what=name)


def test_nemotron_h_parity_all_heads():
    """Full-size Nemotron-H-like workload (8 B/C groups of 16 heads), launched
    exactly as the benchmark launches it; every head of every sequence is
    compared with the oracle, so every group of the grouped B/C map
    (g = h // (nheads / ngroups)) is checked at full size, including the heads
    on both sides of each group edge."""
    w = W.workload("nemotron_h")
    y, pool, _, ws = run_cuda(w)
    import mamba_ssd_chunked_varlen_gb300 as pkg
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    check_all_heads(w, y, pool, what="nemotron_h")


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_small(seed):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.random_small_workload(seed)
    if pkg.ssd_scan_varlen_workspace_size(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups,
                                          w.dstate, w.chunk_size) == 0:
        with pytest.raises(pkg.SSDError):
            run_cuda(w, workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
        return
    _check_full(w, what=f"fuzz{seed}")


@pytest.mark.parametrize("Q", [64, 128, 256])
def test_every_chunk_size(Q):
    w = W.make_workload("q", [700, 129, 1, 256, 64], 8, 64, 2, 128, Q, max_slots=7, seed=31,
                        has_init_p=0.6)
    _check_full(w, what=f"Q={Q}")


@pytest.mark.parametrize("P,N,Q", [(128, 128, 256), (128, 256, 128), (16, 16, 64),
                                   (64, 256, 64), (32, 64, 128)])
def test_shape_corners(P, N, Q):
    w = W.make_workload("corner", [513, 255, 3], 4, P, 2, N, Q, max_slots=4, seed=P + N + Q,
                        has_init_p=0.5)
    _check_full(w, what=f"P={P} N={N} Q={Q}")


def test_empty_optionals():
    w = W.make_workload("opt", [300, 50], 4, 64, 1, 64, 128, max_slots=3, seed=40,
                        with_D=False, with_dt_bias=False)
    w.has_initial_state = None
    _check_full(w, what="optionals")


def test_dt_softplus_off():
    w = W.make_workload("nosp", [400, 33], 4, 64, 2, 64, 128, max_slots=3, seed=41,
                        has_init_p=0.5, dt_softplus=False)
    _check_full(w, what="no softplus")


def test_zero_and_one_length_sequences():
    w = W.make_workload("short", [0, 1, 0, 2, 1, 300, 0], 4, 32, 1, 32, 64, max_slots=9,
                        seed=42, has_init_p=0.5)
    w.has_initial_state[:] = [1, 0, 0, 1, 1, 1, 0]
    _check_full(w, what="short")


def test_total_len_zero_writes_slots():
    w = W.make_workload("empty", [0, 0, 0], 2, 32, 1, 32, 64, max_slots=5, seed=43)
    w.has_initial_state[:] = [1, 0, 1]
    y, pool, _, ws = run_cuda(w)
    import mamba_ssd_chunked_varlen_gb300 as pkg
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    _, pool_ref = recurrence.run_workload(w)
    np.testing.assert_array_equal(pool.cpu().numpy(), pool_ref)


def test_batch_zero_is_a_no_op():
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.make_workload("b0", [10], 2, 32, 1, 32, 64, max_slots=2, seed=44)
    d = to_device(w)
    before = d["ssm_pool"].clone()
    y = torch.zeros_like(d["x"])
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    pkg.ssd_scan_varlen_fwd(y[:0], d["x"][:0], d["dt"][:0], d["A"], d["B"][:0], d["C"][:0],
                            d["D"], d["dt_bias"], d["ssm_pool"], d["query_start_loc"][:1], None,
                            d["cache_indices"][:0], chunk_size=64, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(before, d["ssm_pool"])


def test_bad_cache_index_sets_flag_and_skips_slot():
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.make_workload("badslot", [100, 60], 2, 32, 1, 32, 64, max_slots=3, seed=45)
    w.cache_indices = np.array([1, 7], np.uint32)  # 7 >= max_slots
    y, pool, _, ws = run_cuda(w)
    flags = pkg.ssd_scan_varlen_read_errors(ws)
    assert flags & pkg.binding.DEVERR_BAD_CACHE_INDEX
    pg = pool.cpu().numpy()
    for s in (0, 2):
        assert np.array_equal(pg[s], w.ssm_pool[s])
    # the valid sequence is still correct
    good = W.make_workload("badslot", [100, 60], 2, 32, 1, 32, 64, max_slots=3, seed=45)
    good.cache_indices = np.array([1, 0], np.uint32)
    y_ref, pool_ref = recurrence.run_workload(good)
    check_y(y_to_f64(y), y_ref, rows=slice(0, 100), what="valid sequence")
    rel = np.linalg.norm(pg[1] - pool_ref[1]) / np.linalg.norm(pool_ref[1])
    assert rel < 1e-3


def test_bad_query_start_loc_sets_flag_and_writes_nothing():
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.make_workload("badqsl", [100, 60], 2, 32, 1, 32, 64, max_slots=3, seed=46)
    d = to_device(w)
    d["query_start_loc"] = torch.tensor([0, 120, 90], dtype=torch.int32, device="cuda")
    pool_before = d["ssm_pool"].clone()
    y, pool, _, ws = run_cuda(w, dev=d)
    flags = pkg.ssd_scan_varlen_read_errors(ws)
    assert flags & pkg.binding.DEVERR_BAD_QUERY_START_LOC
    assert torch.equal(pool_before, pool)
    assert torch.isnan(y.float()).all()  # y untouched (was NaN-filled)


@pytest.mark.parametrize("qsl", [[0, 300], [1, 400], [0, 500]])
def test_bad_query_start_loc_one_sequence(qsl):
    """One sequence (whose blocks the kernels place before reading
    query_start_loc): a query_start_loc that does not span [0, total_len]
    still sets the flag and writes nothing."""
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.make_workload("badqsl1", [400], 4, 64, 1, 64, 128, max_slots=2, seed=47,
                        has_init_p=1.0)
    d = to_device(w)
    d["query_start_loc"] = torch.tensor(qsl, dtype=torch.int32, device="cuda")
    pool_before = d["ssm_pool"].clone()
    y, pool, _, ws = run_cuda(w, dev=d)
    flags = pkg.ssd_scan_varlen_read_errors(ws)
    assert flags & pkg.binding.DEVERR_BAD_QUERY_START_LOC
    assert not flags & pkg.binding.DEVERR_TIMEOUT
    assert torch.equal(pool_before, pool)
    assert torch.isnan(y.float()).all()


# ---------------------------------------------------------------- routing, bit-exact

def test_permuting_the_batch_is_bit_exact():
    w = W.workload("ragged")
    y1, pool1, _, _ = run_cuda(w)
    perm = np.random.default_rng(3).permutation(w.batch)
    lens = w.seq_lens
    starts = w.query_start_loc[:-1]
    order = np.concatenate([np.arange(starts[b], starts[b] + lens[b]) for b in perm])
    w2 = W.Workload(name="perm", nheads=w.nheads, head_dim=w.head_dim, ngroups=w.ngroups,
                    dstate=w.dstate, chunk_size=w.chunk_size, x=w.x[order], dt=w.dt[order],
                    A=w.A, B=w.B[order], C=w.C[order], D=w.D, dt_bias=w.dt_bias,
                    ssm_pool=w.ssm_pool,
                    query_start_loc=np.concatenate([[0], np.cumsum(lens[perm])]).astype(np.int32),
                    has_initial_state=w.has_initial_state[perm],
                    cache_indices=w.cache_indices[perm])
    y2, pool2, _, _ = run_cuda(w2)
    y1n = y1.view(torch.int16).cpu().numpy()
    y2n = y2.view(torch.int16).cpu().numpy()
    np.testing.assert_array_equal(y1n[order], y2n)
    np.testing.assert_array_equal(pool1.cpu().numpy().view(np.uint32),
                                  pool2.cpu().numpy().view(np.uint32))


def test_sequence_alone_equals_sequence_in_batch():
    w = W.workload("ragged")
    y, pool, _, _ = run_cuda(w)
    b = 3
    t0, t1 = int(w.query_start_loc[b]), int(w.query_start_loc[b + 1])
    w1 = W.Workload(name="alone", nheads=w.nheads, head_dim=w.head_dim, ngroups=w.ngroups,
                    dstate=w.dstate, chunk_size=w.chunk_size, x=w.x[t0:t1], dt=w.dt[t0:t1],
                    A=w.A, B=w.B[t0:t1], C=w.C[t0:t1], D=w.D, dt_bias=w.dt_bias,
                    ssm_pool=w.ssm_pool, query_start_loc=np.array([0, t1 - t0], np.int32),
                    has_initial_state=w.has_initial_state[b:b + 1],
                    cache_indices=w.cache_indices[b:b + 1])
    ya, poola, _, _ = run_cuda(w1)
    np.testing.assert_array_equal(y.view(torch.int16).cpu().numpy()[t0:t1],
                                  ya.view(torch.int16).cpu().numpy())
    s = int(w.cache_indices[b])
    np.testing.assert_array_equal(pool.cpu().numpy()[s].view(np.uint32),
                                  poola.cpu().numpy()[s].view(np.uint32))


def test_repeated_calls_are_bit_identical():
    w = W.workload("serving_mix")
    y1, p1, _, ws = run_cuda(w)
    y2, p2, _, _ = run_cuda(w, workspace=ws)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(p1.view(torch.int32), p2.view(torch.int32))


def test_runs_on_a_side_stream():
    w = W.workload("tiny")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, pool, _, _ = run_cuda(w, stream=s)
    s.synchronize()
    y_ref, pool_ref = recurrence.run_workload(w)
    check_y(y_to_f64(y), y_ref, what="side stream")
