"""The fused chunk-state walk (chunk states and the inter-chunk state
recurrence in one kernel), which the library takes for calls of long
sequences with many heads whose chunk states would exceed the L2.

Every case first asserts that the library picks the walk for its sizes, so
that these tests exercise it, then compares with the oracle (fp64 per-token
recurrence) on every head, group by group, every sequence: y at the y tolerance,
written slots at the state tolerance, untouched slots byte-identical.  The
cases cover both tensor-memory column widths (64 and 128), two dstate tiles,
64-token chunks, the bf16 pool, the separate-states form, and strided inputs
with dt by TMA and by plain loads (a dt row pitch that is no multiple of 16
bytes).
"""
from __future__ import annotations

import copy

import numpy as np
import pytest

from mamba_ssd_chunked_varlen_gb300 import workloads as W
from oracle import recurrence

from helpers import (STATE_REL_L2, check_all_heads, check_slots, check_y, run_cuda,
                     to_device, y_to_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LENS = [4059, 4196, 4033]   # ragged tails, no length a multiple of 128


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mamba_ssd_chunked_varlen_gb300 as pkg
    from mamba_ssd_chunked_varlen_gb300 import build
    build.build()
    pkg.library()


def _workload(H=128, P=64, G=8, N=128, Q=256, seed=401, init_p=0.7):
    return W.make_workload(f"walk_{H}_{P}_{G}_{N}_{Q}", LENS, H, P, G, N, Q, max_slots=8,
                           seed=seed, has_init_p=init_p)


def _assert_walk(w):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    assert pkg.ssd_scan_varlen_fused_walk(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups,
                                          w.dstate, w.chunk_size), "sizes do not take the walk"


def _head_ranges(w):
    """Head ranges compared with the oracle: every head, one B/C group at a time."""
    hpg = w.nheads // w.ngroups
    return tuple((h, h + hpg) for h in range(0, w.nheads, hpg))


def _check_sampled(w, y, pool, what):
    """Every head of every sequence (one oracle run, compared group by group)."""
    check_all_heads(w, y, pool, what=what)


@pytest.mark.parametrize("shape", [
    dict(),                              # 2 heads per item: 128 columns
    dict(N=256),                         # two 128-row dstate tiles
    dict(P=32),                          # 64-column items
    dict(P=128, G=16),                   # one head of 128 columns per item
    dict(Q=64),                          # 64-token chunks
])
def test_walk_parity_in_place(shape):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = _workload(**shape)
    _assert_walk(w)
    # the walk, chunk scan, short sequences and (a many-wave call) the block map
    assert pkg.ssd_scan_varlen_num_launches(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups,
                                            w.dstate, w.chunk_size) == 4
    y, pool, _, ws = run_cuda(w)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    _check_sampled(w, y, pool, f"walk {shape}")


def test_walk_bf16_pool():
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = _workload(seed=402)
    _assert_walk(w)
    pool_bits = W.f32_to_bf16_bits(w.ssm_pool)
    wr = copy.copy(w)
    wr.ssm_pool = W.bf16_bits_to_f32(pool_bits)   # the bf16 pool's values, exactly
    d = to_device(w)
    pool = torch.from_numpy(pool_bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = pkg.alloc_workspace(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups, w.dstate,
                             w.chunk_size)
    pkg.ssd_scan_varlen_fwd_bf16_pool(y, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                      d["dt_bias"], pool, d["query_start_loc"],
                                      d["has_initial_state"], d["cache_indices"],
                                      chunk_size=w.chunk_size, workspace=ws)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    got_bits = pool.view(torch.int16).cpu().numpy().view(np.uint16)
    got = W.bf16_bits_to_f32(got_bits).astype(np.float64)
    yg = y_to_f64(y)
    written = set(int(s) for s in w.cache_indices)
    y_ref, pool_ref = recurrence.run_workload(wr)
    for heads in _head_ranges(w):
        check_y(yg[:, heads[0]:heads[1]], y_ref[:, heads[0]:heads[1]], what=f"bf16 pool {heads}")
        for s in written:
            ref = pool_ref[s][heads[0]:heads[1]].astype(np.float64)
            g = got[s][heads[0]:heads[1]]
            rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
            # the fp32 bar plus one bf16 rounding of the stored state
            assert rel <= STATE_REL_L2 + 2.0 ** -8, f"bf16 pool slot {s} heads {heads}: {rel:.3e}"
    for s in range(w.ssm_pool.shape[0]):
        if s not in written:
            assert np.array_equal(got_bits[s], pool_bits[s]), f"untouched slot {s} changed"


def test_walk_states_form():
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = _workload(seed=403, init_p=0.0)
    _assert_walk(w)
    rng = np.random.default_rng(404)
    init = (rng.standard_normal((w.batch, w.nheads, w.head_dim, w.dstate)) * 0.1).astype(np.float32)
    flags = np.array([1, 0, 1], dtype=np.uint8)
    d = to_device(w)
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    init_t = torch.from_numpy(init).cuda()
    final = torch.full(init.shape, float("nan"), dtype=torch.float32, device="cuda")
    ws = pkg.alloc_workspace(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups, w.dstate,
                             w.chunk_size)
    pkg.ssd_scan_varlen_fwd_states(y, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                   d["dt_bias"], init_t, torch.from_numpy(flags).cuda(), final,
                                   d["query_start_loc"], chunk_size=w.chunk_size, workspace=ws)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    # the oracle on the in-place form: slot cache_indices[b] holds initial_states[b]
    wr = copy.copy(w)
    wr.has_initial_state = flags
    wr.ssm_pool = np.zeros_like(w.ssm_pool)
    wr.ssm_pool[np.asarray(w.cache_indices, dtype=np.int64)] = init
    yg = y_to_f64(y)
    fin = final.cpu().numpy()
    assert np.all(np.isfinite(fin)), "final_states not fully written"
    y_ref, pool_ref = recurrence.run_workload(wr)
    for heads in _head_ranges(w):
        check_y(yg[:, heads[0]:heads[1]], y_ref[:, heads[0]:heads[1]], what=f"states {heads}")
        for b, s in enumerate(w.cache_indices):
            ref = pool_ref[int(s)][heads[0]:heads[1]].astype(np.float64)
            g = fin[b][heads[0]:heads[1]].astype(np.float64)
            rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
            assert rel <= STATE_REL_L2, f"states: sequence {b} heads {heads}: {rel:.3e}"


@pytest.mark.parametrize("dt_pitch_extra", [7, 8])
def test_walk_strided_inputs(dt_pitch_extra):
    """x, B, C as column slices of one wide buffer; dt in a buffer of its own
    whose row pitch is H + 7 (no multiple of 16 bytes: plain loads) or H + 8
    (TMA)."""
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = _workload(seed=405)
    _assert_walk(w)
    d = to_device(w)
    T, H, P, G, N = w.total_len, w.nheads, w.head_dim, w.ngroups, w.dstate
    pad = 8
    o_b = pad + H * P + pad
    o_c = o_b + G * N
    width = o_c + G * N + pad
    buf = torch.full((T, width), float("nan"), dtype=torch.bfloat16, device="cuda")
    buf[:, pad:pad + H * P] = d["x"].reshape(T, H * P)
    buf[:, o_b:o_c] = d["B"].reshape(T, G * N)
    buf[:, o_c:o_c + G * N] = d["C"].reshape(T, G * N)
    dbuf = torch.full((T, H + dt_pitch_extra), float("nan"), dtype=torch.bfloat16, device="cuda")
    dbuf[:, :H] = d["dt"]
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = pkg.alloc_workspace(T, w.batch, H, P, G, N, w.chunk_size)
    pkg.ssd_scan_varlen_fwd_strided(y, buf[:, pad:pad + H * P].unflatten(1, (H, P)), dbuf[:, :H],
                                    d["A"], buf[:, o_b:o_c].unflatten(1, (G, N)),
                                    buf[:, o_c:o_c + G * N].unflatten(1, (G, N)), d["D"],
                                    d["dt_bias"], d["ssm_pool"], d["query_start_loc"],
                                    d["has_initial_state"], d["cache_indices"],
                                    chunk_size=w.chunk_size, workspace=ws)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    _check_sampled(w, y, d["ssm_pool"], f"strided dt pitch H+{dt_pitch_extra}")


def _sub(w, lo, hi):
    """Sequences [lo, hi) of `w` as a workload of their own (same slots)."""
    import dataclasses
    t0, t1 = int(w.query_start_loc[lo]), int(w.query_start_loc[hi])
    return dataclasses.replace(
        w, x=w.x[t0:t1], dt=w.dt[t0:t1], B=w.B[t0:t1], C=w.C[t0:t1],
        query_start_loc=(w.query_start_loc[lo:hi + 1] - t0).astype(np.int32),
        has_initial_state=w.has_initial_state[lo:hi], cache_indices=w.cache_indices[lo:hi])


def test_walk_with_block_table():
    """514 sequences of 2049-2199 tokens: the block-map kernel lists the
    sequences and the walk reads its list.  Every sequence must give the bits
    it gives in a call of 257 (where each walking CTA lists them itself), and
    sampled sequences must match the oracle."""
    import dataclasses
    import mamba_ssd_chunked_varlen_gb300 as pkg
    rng = np.random.default_rng(406)
    lens = [int(v) for v in rng.integers(2049, 2200, size=514)]
    w = W.make_workload("walk_table", lens, 8, 16, 1, 64, 256, max_slots=520, seed=407,
                        has_init_p=0.5)
    _assert_walk(w)
    assert pkg.ssd_scan_varlen_num_launches(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups,
                                            w.dstate, w.chunk_size) == 4
    y, pool, _, ws = run_cuda(w)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    parts = [_sub(w, 0, 257), _sub(w, 257, 514)]
    for part in parts:
        _assert_walk(part)
    y1, pool1, _, _ = run_cuda(parts[0])
    w2 = dataclasses.replace(parts[1], ssm_pool=pool1.cpu().numpy())
    y2, pool2, _, _ = run_cuda(w2)
    t_cut = int(w.query_start_loc[257])
    assert torch.equal(y[:t_cut].view(torch.int16), y1.view(torch.int16))
    assert torch.equal(y[t_cut:].view(torch.int16), y2.view(torch.int16))
    assert torch.equal(pool.view(torch.int32), pool2.view(torch.int32))
    # the oracle on the first and the last two sequences
    yg = y_to_f64(y)
    pg = pool.cpu().numpy()
    for lo, hi in ((0, 2), (512, 514)):
        ws_ = _sub(w, lo, hi)
        y_ref, pool_ref = recurrence.run_workload(ws_)
        t0, t1 = int(w.query_start_loc[lo]), int(w.query_start_loc[hi])
        check_y(yg[t0:t1], y_ref, what=f"sequences [{lo}, {hi})")
        for b in range(lo, hi):
            s = int(w.cache_indices[b])
            ref = pool_ref[s].astype(np.float64)
            rel = np.linalg.norm(pg[s] - ref) / np.linalg.norm(ref)
            assert rel <= STATE_REL_L2, f"sequence {b} slot {s}: {rel:.3e}"


def test_walk_with_short_and_empty_sequences():
    """A walk call may hold sequences short enough for the per-token kernel
    (and empty ones): they are not walked, their slots are still written."""
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = W.make_workload("walk_mix", [4100, 0, 5, 4200, 4000], 128, 64, 8, 128, 256, max_slots=8,
                        seed=408, has_init_p=0.6)
    _assert_walk(w)
    y, pool, _, ws = run_cuda(w)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    _check_sampled(w, y, pool, "walk with short sequences")


def test_walk_bad_query_start_loc():
    """A decreasing query_start_loc: the flag is set, nothing is written."""
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = _workload(seed=409)
    _assert_walk(w)
    d = to_device(w)
    qsl = w.query_start_loc.copy()
    qsl[1] = qsl[2] + 1                 # a negative length
    d["query_start_loc"] = torch.from_numpy(qsl).cuda()
    pool_before = d["ssm_pool"].clone()
    y, pool, _, ws = run_cuda(w, dev=d)
    flags = pkg.ssd_scan_varlen_read_errors(ws)
    assert flags & pkg.binding.DEVERR_BAD_QUERY_START_LOC
    assert not flags & pkg.binding.DEVERR_TIMEOUT
    assert torch.equal(pool_before, pool)
    assert torch.isnan(y.float()).all()


def test_walk_bad_cache_index():
    """A cache index past the pool: the flag is set, that sequence's slot
    access is skipped (zero initial state, no write-back), the others are
    computed as usual."""
    import mamba_ssd_chunked_varlen_gb300 as pkg
    w = _workload(seed=410)
    _assert_walk(w)
    w.cache_indices = np.array([w.cache_indices[0], 11, w.cache_indices[2]], np.uint32)
    y, pool, _, ws = run_cuda(w)
    flags = pkg.ssd_scan_varlen_read_errors(ws)
    assert flags & pkg.binding.DEVERR_BAD_CACHE_INDEX
    assert not flags & pkg.binding.DEVERR_TIMEOUT
    pg = pool.cpu().numpy()
    # the oracle with sequence 1 starting from zero and writing a spare slot
    wr = copy.copy(w)
    wr.ssm_pool = np.concatenate([w.ssm_pool, np.zeros_like(w.ssm_pool[:1])])
    spare = w.ssm_pool.shape[0]
    wr.cache_indices = np.array([w.cache_indices[0], spare, w.cache_indices[2]], np.uint32)
    wr.has_initial_state = w.has_initial_state.copy()
    wr.has_initial_state[1] = 0
    yg = y_to_f64(y)
    y_ref, pool_ref = recurrence.run_workload(wr)
    for heads in _head_ranges(w):
        check_y(yg[:, heads[0]:heads[1]], y_ref[:, heads[0]:heads[1]], what=f"bad slot {heads}")
        for b in (0, 2):
            s = int(w.cache_indices[b])
            ref = pool_ref[s][heads[0]:heads[1]].astype(np.float64)
            rel = np.linalg.norm(pg[s][heads[0]:heads[1]] - ref) / np.linalg.norm(ref)
            assert rel <= STATE_REL_L2, f"bad slot: sequence {b} heads {heads}: {rel:.3e}"
    written = {int(w.cache_indices[0]), int(w.cache_indices[2])}
    for s in range(w.ssm_pool.shape[0]):
        if s not in written:
            assert np.array_equal(pg[s].view(np.uint32), w.ssm_pool[s].view(np.uint32)), \
                f"slot {s} changed"


@pytest.mark.parametrize("variant", ["empty_optionals", "softplus_off"])
def test_walk_optionals_and_softplus(variant):
    """No D, no dt_bias and no has_initial_state (zero initial states), or dt
    used as given (dt + dt_bias, no softplus)."""
    import mamba_ssd_chunked_varlen_gb300 as pkg
    if variant == "empty_optionals":
        w = W.make_workload("walk_noopt", LENS, 128, 64, 8, 128, 256, max_slots=8, seed=411,
                            with_D=False, with_dt_bias=False)
        w.has_initial_state = None
    else:
        w = W.make_workload("walk_nosp", LENS, 128, 64, 8, 128, 256, max_slots=8, seed=412,
                            has_init_p=0.7, dt_softplus=False)
    _assert_walk(w)
    y, pool, _, ws = run_cuda(w)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    _check_sampled(w, y, pool, f"walk {variant}")


# (heads, head_dim, groups, dstate, chunk, lengths, options): sizes that take
# the walk with every instantiation and tile count: 128 or 64 columns per item,
# one to eight heads per item, one or two dstate tiles (144: a mostly empty
# second tile), 64- to 256-token chunks, 1 to 16 groups, a short sequence
# beside the long ones, empty optionals and softplus off
WALK_SHAPES = [
    (64, 128, 4, 128, 128, [4100, 5003, 3900, 4500], {}),
    (96, 32, 3, 256, 256, [2500, 3000, 2100, 2900, 2600], {}),
    (256, 16, 16, 144, 64, [2050, 2600, 3100], {}),
    (128, 64, 1, 64, 256, [6000, 7000], {"with_D": False}),
    (80, 64, 5, 256, 128, [3000, 4000, 2500, 7], {}),
    (128, 64, 8, 128, 256, [3000, 3500, 2900, 2700], {"dt_softplus": False, "with_dt_bias": False}),
]


@pytest.mark.parametrize("case", range(len(WALK_SHAPES)))
def test_walk_shapes(case):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    H, P, G, N, Q, lens, opts = WALK_SHAPES[case]
    w = W.make_workload(f"walk_shape{case}", lens, H, P, G, N, Q, max_slots=len(lens) + 3,
                        seed=420 + case, has_init_p=0.6, **opts)
    _assert_walk(w)
    y, pool, _, ws = run_cuda(w)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    _check_sampled(w, y, pool, f"walk shape {case}")
