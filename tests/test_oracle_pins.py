"""Pins for the CPU oracle (no GPU).

The oracle is the per-token recurrence of the Modular page "mamba2_ssd_scan"
("Per-token recurrence") in fp64.  The pages print no worked example, so it is
pinned by things other than itself:

* hand-worked cases with exact values (tests/golden/hand_worked.json);
* brute force: the materialised quadratic form on small inputs;
* the chunked form of the kernelindex page "Mamba chunk scan with segsum" at
  several chunk sizes (the module page states the two forms agree);
* closed forms: the single-token result, A = 0 (a plain prefix sum, checked
  against numpy.cumsum), C = 0 (y = D x), a memoryless limit;
* invariants: concatenation / reset at query_start_loc boundaries, split
  prefill continuation through a pool slot, initial-state linearity, grouped
  B/C equal to replicated B/C, empty optionals equal to zeros, untouched slots;
* mutation: each plausible slip planted in a copy of the oracle's C source
  makes at least one of these checks fail.
"""
from __future__ import annotations

import json
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import recurrence, quadratic, chunked
from mamba_ssd_chunked_varlen_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def kwargs(w):
    return dict(x=w.x, dt=w.dt, A=w.A, B=w.B, C=w.C, D=w.D, dt_bias=w.dt_bias,
                ssm_pool=w.ssm_pool, query_start_loc=w.query_start_loc,
                has_initial_state=w.has_initial_state, cache_indices=w.cache_indices,
                dt_softplus=w.dt_softplus)


def rel_max(a, b):
    m = max(np.abs(b).max(), 1e-300) if b.size else 1.0
    return float(np.abs(a - b).max() / m) if a.size else 0.0


def written_slots(w):
    return sorted(set(int(s) for s in w.cache_indices))


def bf16(a):
    return W.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


# ----------------------------------------------------------------------------
# hand-worked golden cases

def _golden_cases():
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_golden(case):
    f32 = lambda v: None if v is None else np.asarray(v, dtype=np.float32)
    y, pool = recurrence.ssd_varlen_fwd(
        x=bf16(case["x"]), dt=bf16(case["dt"]), A=f32(case["A"]), B=bf16(case["B"]),
        C=bf16(case["C"]), D=f32(case["D"]), dt_bias=f32(case["dt_bias"]),
        ssm_pool=f32(case["pool"]),
        query_start_loc=np.asarray(case["query_start_loc"], np.int32),
        has_initial_state=np.asarray(case["has_initial_state"], np.uint8),
        cache_indices=np.asarray(case["cache_indices"], np.uint32),
        dt_softplus=case["dt_softplus"])
    np.testing.assert_allclose(y, np.asarray(case["expected_y"]), rtol=1e-15, atol=0)
    np.testing.assert_array_equal(pool, np.asarray(case["expected_pool"], dtype=np.float32))


# ----------------------------------------------------------------------------
# brute force and chunked forms

def test_recurrence_vs_quadratic_tiny():
    w = W.workload("tiny")
    y, pool = recurrence.run_workload(w)
    yq, pq = quadratic.ssd_varlen_fwd(**kwargs(w))
    assert rel_max(y, yq) < 1e-12
    for s in written_slots(w):
        assert rel_max(pool[s], pq[s]) < 1e-6  # both are fp32 roundings of fp64 states


@pytest.mark.parametrize("seed", range(8))
def test_recurrence_vs_quadratic_fuzz(seed):
    w = W.random_small_workload(seed, max_total=400)
    y, pool = recurrence.run_workload(w)
    yq, pq = quadratic.ssd_varlen_fwd(**kwargs(w))
    assert rel_max(y, yq) < 1e-11
    for s in written_slots(w):
        np.testing.assert_allclose(pool[s], pq[s], rtol=1e-6, atol=1e-7 * np.abs(pq[s]).max())


@pytest.mark.parametrize("Q", [1, 7, 64, 256, 4096])
def test_chunk_size_invariance(Q):
    w = W.make_workload("inv", [300, 1, 0, 257, 150], nheads=4, head_dim=16, ngroups=2,
                        dstate=24, chunk_size=Q, max_slots=6, seed=11, has_init_p=0.6)
    y, pool = recurrence.run_workload(w)
    yc, pc = chunked.ssd_varlen_fwd(**kwargs(w), chunk_size=Q)
    assert rel_max(y, yc) < 1e-12
    for s in written_slots(w):
        np.testing.assert_allclose(pool[s], pc[s], rtol=1e-6, atol=1e-7 * np.abs(pc[s]).max())


# ----------------------------------------------------------------------------
# closed forms

@pytest.mark.parametrize("with_init", [False, True])
@pytest.mark.parametrize("softplus", [True, False])
def test_single_token_closed_form(with_init, softplus):
    rng = np.random.default_rng(5)
    H, P, G, N = 4, 8, 2, 16
    w = W.make_workload("one", [1, 1, 1], H, P, G, N, 64, max_slots=3, seed=3,
                        has_init_p=1.0 if with_init else 0.0, dt_softplus=softplus)
    y, pool = recurrence.run_workload(w)
    X = W.bf16_bits_to_f32(w.x).astype(np.float64)
    DT = W.bf16_bits_to_f32(w.dt).astype(np.float64)
    Bf = W.bf16_bits_to_f32(w.B).astype(np.float64)
    Cf = W.bf16_bits_to_f32(w.C).astype(np.float64)
    for t in range(3):
        slot = int(w.cache_indices[t])
        for h in range(H):
            g = h // (H // G)
            v = DT[t, h] + float(w.dt_bias[h])
            d = np.logaddexp(0.0, v) if softplus else v
            S0 = w.ssm_pool[slot, h].astype(np.float64) if with_init else np.zeros((P, N))
            S = np.exp(float(w.A[h]) * d) * S0 + d * np.outer(X[t, h], Bf[t, g])
            y_exp = S @ Cf[t, g] + float(w.D[h]) * X[t, h]
            if not with_init:
                # y = (C . (dt B)) x + D x
                y_exp2 = (Cf[t, g] @ (d * Bf[t, g])) * X[t, h] + float(w.D[h]) * X[t, h]
                np.testing.assert_allclose(y_exp, y_exp2, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(y[t, h], y_exp, rtol=1e-13, atol=1e-13)
            np.testing.assert_array_equal(pool[slot, h], S.astype(np.float32))


def test_A_zero_is_prefix_sum():
    w = W.make_workload("a0", [200, 57], 2, 8, 1, 12, 64, max_slots=2, seed=4, has_init_p=1.0)
    w.A[:] = 0.0
    y, pool = recurrence.run_workload(w)
    X = W.bf16_bits_to_f32(w.x).astype(np.float64)
    DT = W.bf16_bits_to_f32(w.dt).astype(np.float64)
    Bf = W.bf16_bits_to_f32(w.B).astype(np.float64)
    Cf = W.bf16_bits_to_f32(w.C).astype(np.float64)
    qsl = w.query_start_loc
    for b in range(2):
        t0, t1 = qsl[b], qsl[b + 1]
        slot = int(w.cache_indices[b])
        for h in range(2):
            d = np.logaddexp(0.0, DT[t0:t1, h] + float(w.dt_bias[h]))
            upd = d[:, None, None] * X[t0:t1, h][:, :, None] * Bf[t0:t1, 0][:, None, :]
            S = np.cumsum(upd, axis=0) + w.ssm_pool[slot, h].astype(np.float64)[None]
            y_exp = np.einsum("tpn,tn->tp", S, Cf[t0:t1, 0]) + float(w.D[h]) * X[t0:t1, h]
            np.testing.assert_allclose(y[t0:t1, h], y_exp, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(pool[slot, h], S[-1], rtol=1e-6)


def test_C_zero_gives_D_skip_exactly():
    w = W.make_workload("c0", [100, 33], 4, 8, 2, 8, 64, max_slots=2, seed=6, has_init_p=0.5)
    w.C[:] = 0
    y, _ = recurrence.run_workload(w)
    X = W.bf16_bits_to_f32(w.x).astype(np.float64)
    np.testing.assert_array_equal(y, w.D.astype(np.float64)[None, :, None] * X)


def test_strongly_negative_A_is_memoryless():
    w = W.make_workload("neg", [64], 2, 8, 1, 16, 64, max_slots=1, seed=8)
    w.A[:] = -1e6
    y, pool = recurrence.run_workload(w)
    X = W.bf16_bits_to_f32(w.x).astype(np.float64)
    DT = W.bf16_bits_to_f32(w.dt).astype(np.float64)
    Bf = W.bf16_bits_to_f32(w.B).astype(np.float64)
    Cf = W.bf16_bits_to_f32(w.C).astype(np.float64)
    for h in range(2):
        d = np.logaddexp(0.0, DT[:, h] + float(w.dt_bias[h]))
        cb = np.einsum("tn,tn->t", Cf[:, 0], Bf[:, 0])
        y_exp = (d * cb)[:, None] * X[:, h] + float(w.D[h]) * X[:, h]
        np.testing.assert_allclose(y[:, h], y_exp, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# invariants

def test_concatenation_equals_separate_runs():
    w = W.make_workload("cat", [190, 75, 1], 4, 16, 2, 16, 64, max_slots=5, seed=9,
                        has_init_p=0.7)
    y, pool = recurrence.run_workload(w)
    qsl = w.query_start_loc
    for b in range(3):
        t0, t1 = int(qsl[b]), int(qsl[b + 1])
        yb, pb = recurrence.ssd_varlen_fwd(
            x=w.x[t0:t1], dt=w.dt[t0:t1], A=w.A, B=w.B[t0:t1], C=w.C[t0:t1], D=w.D,
            dt_bias=w.dt_bias, ssm_pool=w.ssm_pool,
            query_start_loc=np.array([0, t1 - t0], np.int32),
            has_initial_state=w.has_initial_state[b:b + 1],
            cache_indices=w.cache_indices[b:b + 1])
        np.testing.assert_array_equal(y[t0:t1], yb)
        s = int(w.cache_indices[b])
        np.testing.assert_array_equal(pool[s], pb[s])


def test_split_prefill_continuation():
    w = W.make_workload("split", [333], 2, 16, 1, 32, 64, max_slots=2, seed=10)
    y, pool = recurrence.run_workload(w)
    k = 120
    s = int(w.cache_indices[0])
    y1, p1 = recurrence.ssd_varlen_fwd(
        x=w.x[:k], dt=w.dt[:k], A=w.A, B=w.B[:k], C=w.C[:k], D=w.D, dt_bias=w.dt_bias,
        ssm_pool=w.ssm_pool, query_start_loc=np.array([0, k], np.int32),
        has_initial_state=np.array([0], np.uint8), cache_indices=w.cache_indices)
    y2, p2 = recurrence.ssd_varlen_fwd(
        x=w.x[k:], dt=w.dt[k:], A=w.A, B=w.B[k:], C=w.C[k:], D=w.D, dt_bias=w.dt_bias,
        ssm_pool=p1, query_start_loc=np.array([0, 333 - k], np.int32),
        has_initial_state=np.array([1], np.uint8), cache_indices=w.cache_indices)
    np.testing.assert_array_equal(y[:k], y1[:k])
    # the only difference is the fp32 rounding of the state stored in the slot
    assert rel_max(y2, y[k:]) < 1e-6
    assert rel_max(p2[s], pool[s]) < 1e-6


def test_initial_state_linearity():
    w = W.make_workload("lin", [150], 2, 8, 1, 16, 64, max_slots=3, seed=12, has_init_p=1.0)
    rng = np.random.default_rng(0)
    # dyadic values, so that S1 + S2 is exact in the fp32 pool
    S1 = (rng.integers(-64, 65, w.ssm_pool.shape[1:]) / 16.0).astype(np.float32)
    S2 = (rng.integers(-64, 65, w.ssm_pool.shape[1:]) / 16.0).astype(np.float32)
    slot = int(w.cache_indices[0])

    def run(S0):
        pool = np.zeros_like(w.ssm_pool)
        pool[slot] = S0
        kw = kwargs(w)
        kw["ssm_pool"] = pool
        kw["has_initial_state"] = np.array([1], np.uint8)
        return recurrence.ssd_varlen_fwd(**kw)

    y0, _ = run(np.zeros_like(S1))
    ya, _ = run(S1)
    yb, _ = run(S2)
    yab, _ = run(S1 + S2)
    np.testing.assert_allclose(yab - y0, (ya - y0) + (yb - y0), rtol=0, atol=1e-9)
    # final state: S_L(S0) - S_L(0) = exp(sum a) S0, per head
    DT = W.bf16_bits_to_f32(w.dt).astype(np.float64)
    kw = kwargs(w)
    kw["ssm_pool"] = np.zeros_like(w.ssm_pool)
    kw["has_initial_state"] = np.array([1], np.uint8)
    kw["ssm_pool"][slot] = S1
    _, pS = recurrence.ssd_varlen_fwd(**kw)
    kw["ssm_pool"] = np.zeros_like(w.ssm_pool)
    _, p0 = recurrence.ssd_varlen_fwd(**kw)
    for h in range(2):
        d = np.logaddexp(0.0, DT[:, h] + float(w.dt_bias[h]))
        decay = np.exp(float(w.A[h]) * d.sum())
        np.testing.assert_allclose(pS[slot, h].astype(np.float64) - p0[slot, h],
                                   decay * S1[h], rtol=0, atol=3e-7 * max(1.0, np.abs(p0).max()))


def test_x_linearity_without_initial_state():
    w = W.make_workload("xlin", [90], 2, 8, 1, 8, 64, max_slots=1, seed=13)
    w.D = None
    y, _ = recurrence.run_workload(w)
    # x -> 2x doubles y exactly (scaling by 2 is exact in bf16 and fp64)
    x2 = W.f32_to_bf16_bits(2.0 * W.bf16_bits_to_f32(w.x))
    kw = kwargs(w)
    kw["x"] = x2
    y2, _ = recurrence.ssd_varlen_fwd(**kw)
    np.testing.assert_array_equal(y2, 2.0 * y)


def test_grouped_equals_replicated():
    w = W.make_workload("grp", [120, 40], 6, 8, 2, 16, 64, max_slots=2, seed=14, has_init_p=0.5)
    y, pool = recurrence.run_workload(w)
    rep = np.arange(6) // 3
    kw = kwargs(w)
    kw["B"] = np.ascontiguousarray(w.B[:, rep])
    kw["C"] = np.ascontiguousarray(w.C[:, rep])
    y2, pool2 = recurrence.ssd_varlen_fwd(**kw)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(pool, pool2)


def test_empty_optionals_equal_zeros():
    w = W.make_workload("opt", [70, 10], 2, 8, 1, 8, 64, max_slots=2, seed=15)
    kw = kwargs(w)
    kw.update(D=None, dt_bias=None, has_initial_state=None)
    y1, p1 = recurrence.ssd_varlen_fwd(**kw)
    kw.update(D=np.zeros(2, np.float32), dt_bias=np.zeros(2, np.float32),
              has_initial_state=np.zeros(2, np.uint8))
    y2, p2 = recurrence.ssd_varlen_fwd(**kw)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(p1, p2)


def test_zero_length_sequence_writes_its_slot():
    w = W.make_workload("zero", [5, 0, 0, 3], 2, 4, 1, 4, 64, max_slots=6, seed=16)
    w.has_initial_state[:] = [0, 1, 0, 0]
    _, pool = recurrence.run_workload(w)
    s1, s2 = int(w.cache_indices[1]), int(w.cache_indices[2])
    np.testing.assert_array_equal(pool[s1], w.ssm_pool[s1])      # initial state written back
    np.testing.assert_array_equal(pool[s2], np.zeros_like(pool[s2]))  # zeros written


def test_untouched_slots_unchanged():
    w = W.workload("ragged")
    w2 = W.make_workload("few", [40, 17, 90], 16, 8, 1, 16, 64, max_slots=64, seed=2,
                         has_init_p=0.5)
    _, pool = recurrence.run_workload(w2)
    touched = set(int(s) for s in w2.cache_indices)
    for s in range(w2.max_slots):
        if s not in touched:
            np.testing.assert_array_equal(pool[s], w2.ssm_pool[s])
    assert w.batch == 8 and all(int(n) % 256 != 0 for n in w.seq_lens)


def test_thread_count_does_not_change_results():
    w = W.make_workload("thr", [100, 60, 7], 8, 8, 2, 16, 64, max_slots=4, seed=17,
                        has_init_p=0.5)
    y1, p1 = recurrence.run_workload(w, num_threads=1)
    y4, p4 = recurrence.run_workload(w, num_threads=4)
    np.testing.assert_array_equal(y1, y4)
    np.testing.assert_array_equal(p1, p4)


def test_head_and_sequence_selection():
    w = W.make_workload("sel", [50, 20, 30], 4, 8, 2, 8, 64, max_slots=3, seed=18,
                        has_init_p=0.5)
    y, pool = recurrence.run_workload(w)
    sel = np.array([1, 0, 1], np.uint8)
    ys, ps = recurrence.run_workload(w, seq_select=sel, heads=(1, 3))
    qsl = w.query_start_loc
    for b in (0, 2):
        t0, t1 = qsl[b], qsl[b + 1]
        np.testing.assert_array_equal(ys[t0:t1, 1:3], y[t0:t1, 1:3])
        s = int(w.cache_indices[b])
        np.testing.assert_array_equal(ps[s, 1:3], pool[s, 1:3])


def test_rejects_bad_arguments():
    w = W.make_workload("bad", [10, 5], 2, 4, 1, 4, 64, max_slots=2, seed=19)
    kw = kwargs(w)
    kw["query_start_loc"] = np.array([0, 12, 14], np.int32)  # does not end at total_len
    with pytest.raises(ValueError):
        recurrence.ssd_varlen_fwd(**kw)
    kw = kwargs(w)
    kw["cache_indices"] = np.array([0, 7], np.uint32)  # slot out of range
    with pytest.raises(ValueError):
        recurrence.ssd_varlen_fwd(**kw)


# ----------------------------------------------------------------------------
# mutation: plant plausible slips in a copy of the oracle and check the pins catch each

MUTANTS = {
    "drop_D": ("acc + Dh * xt[p]", "acc"),
    "exp_sign": ("exp(Ah * d)", "exp(-Ah * d)"),
    "no_softplus": ("dt_softplus ? softplus_f64(v) : v", "v"),
    "drop_bias": ("bf16_to_f64(dt[t * H + h]) + bias", "bf16_to_f64(dt[t * H + h])"),
    "group_index": ("h / heads_per_group", "h % G"),
    "B_C_swapped": ("Sp[n] * dA + dx * Bt[n]", "Sp[n] * dA + dx * Ct[n]"),
    "dt_not_on_input": ("const double dx = d * xt[p];", "const double dx = xt[p];"),
    "init_ignored": ("init ? (double)slot_h[i] : 0.0", "0.0"),
    "output_before_update": ("Sp[n] = Sp[n] * dA + dx * Bt[n];\n                        acc += Ct[n] * Sp[n];",
                             "acc += Ct[n] * Sp[n];\n                        Sp[n] = Sp[n] * dA + dx * Bt[n];"),
    "softplus_log_not_log1p": ("log1p(exp(-fabs(v)))", "log(exp(-fabs(v)))"),
}


def _pin_battery(mod):
    """Cheap pin checks run against a (possibly mutated) oracle module.
    Returns the names of the checks that fail."""
    fails = []
    # golden
    for case in _golden_cases():
        f32 = lambda v: None if v is None else np.asarray(v, dtype=np.float32)
        y, pool = mod.ssd_varlen_fwd(
            x=bf16(case["x"]), dt=bf16(case["dt"]), A=f32(case["A"]), B=bf16(case["B"]),
            C=bf16(case["C"]), D=f32(case["D"]), dt_bias=f32(case["dt_bias"]),
            ssm_pool=f32(case["pool"]),
            query_start_loc=np.asarray(case["query_start_loc"], np.int32),
            has_initial_state=np.asarray(case["has_initial_state"], np.uint8),
            cache_indices=np.asarray(case["cache_indices"], np.uint32),
            dt_softplus=case["dt_softplus"])
        if not (np.allclose(y, case["expected_y"], rtol=1e-15, atol=0)
                and np.array_equal(pool, np.asarray(case["expected_pool"], np.float32))):
            fails.append("golden:" + case["name"])
    # brute force on a grouped, initial-state, ragged case
    w = W.make_workload("mut", [40, 1, 25], 4, 4, 2, 8, 64, max_slots=4, seed=21,
                        has_init_p=0.7)
    w.has_initial_state[:] = [1, 0, 1]
    y, pool = mod.ssd_varlen_fwd(**kwargs(w))
    yq, pq = quadratic.ssd_varlen_fwd(**kwargs(w))
    if rel_max(y, yq) > 1e-11:
        fails.append("quadratic:y")
    if any(rel_max(pool[s], pq[s]) > 1e-6 for s in written_slots(w)):
        fails.append("quadratic:state")
    return fails


class _MutantModule:
    def __init__(self, path):
        import ctypes
        self._lib = ctypes.CDLL(path)
        f = self._lib.ssd_oracle_varlen_fwd
        f.restype = ctypes.c_int
        f.argtypes = recurrence.lib().ssd_oracle_varlen_fwd.argtypes

    def ssd_varlen_fwd(self, **kw):
        saved = recurrence._lib
        recurrence._lib = self._lib
        try:
            return recurrence.ssd_varlen_fwd(**kw)
        finally:
            recurrence._lib = saved


def test_pin_battery_passes_on_the_oracle():
    assert _pin_battery(recurrence) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    src_path = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")
    src = open(src_path).read()
    old, new = MUTANTS[name]
    old_n = " ".join(old.split())
    # match on whitespace-normalised text so indentation does not matter
    import re
    pattern = r"\s+".join(re.escape(tok) for tok in old_n.split(" "))
    mutated, count = re.subn(pattern, new.replace("\\", "\\\\"), src, count=1)
    assert count == 1, f"mutation site for {name} not found"
    c_path = tmp_path / "mut.c"
    c_path.write_text(mutated)
    so_path = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
                    "-shared", str(c_path), "-o", str(so_path), "-lm"], check=True)
    fails = _pin_battery(_MutantModule(str(so_path)))
    assert fails, f"planted mistake {name} was not caught by any pin"
