"""bf16 slot-pool storage (ssd_scan_varlen_fwd_bf16_pool).

"Mamba2SSDChunkScanVarlenFwdInplace" ("Tensor shapes") allows a bf16 ssm_pool
as storage dtype only: the scan accumulates in fp32.  So the expected values
are the oracle's on the same (bf16-valued) initial states, with the final
states then rounded once to bf16.  Tolerance for a written slot: relative L2
<= 1e-3 (the fp32 state bar) + 2^-8 (one bf16 rounding: |bf16(v) - v| <=
2^-8 |v| element-wise); y as for the fp32 pool; every other slot bit-identical.
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

BF16_STATE_REL_L2 = STATE_REL_L2 + 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mamba_ssd_chunked_varlen_gb300 as pkg
    from mamba_ssd_chunked_varlen_gb300 import build
    build.build()
    pkg.library()


@pytest.mark.parametrize("name", ["ragged", "small", "short"])
def test_bf16_pool_parity(name):
    import mamba_ssd_chunked_varlen_gb300 as pkg
    if name == "ragged":
        w = W.workload("ragged")
    elif name == "small":
        w = W.make_workload("bf16pool_small", [300, 1, 129, 64], 6, 32, 2, 64, 64, max_slots=6,
                            seed=97, has_init_p=0.5)
    else:
        w = W.make_workload("bf16pool_short", [0, 5, 0, 200, 1], 4, 64, 1, 128, 128, max_slots=7,
                            seed=98, has_init_p=0.5)
    pool_bits = W.f32_to_bf16_bits(w.ssm_pool)            # the bf16 pool the caller holds
    wr = copy.copy(w)
    wr.ssm_pool = W.bf16_bits_to_f32(pool_bits)           # the same values, exactly, in fp32
    y_ref, pool_ref = recurrence.run_workload(wr)

    d = to_device(w)
    pool = torch.from_numpy(pool_bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    y = torch.full(w.x.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = pkg.alloc_workspace(w.total_len, w.batch, w.nheads, w.head_dim, w.ngroups, w.dstate,
                             w.chunk_size)
    pkg.ssd_scan_varlen_fwd_bf16_pool(y, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                      d["dt_bias"], pool, d["query_start_loc"],
                                      d["has_initial_state"], d["cache_indices"],
                                      chunk_size=w.chunk_size, dt_softplus=w.dt_softplus,
                                      workspace=ws)
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    check_y(y_to_f64(y), y_ref, what=f"bf16 pool {name}")
    got_bits = pool.view(torch.int16).cpu().numpy().view(np.uint16)
    got = W.bf16_bits_to_f32(got_bits).astype(np.float64)
    written = set(int(s) for s in w.cache_indices)
    for s in range(w.ssm_pool.shape[0]):
        if s in written:
            ref = pool_ref[s].astype(np.float64)
            nrm = np.linalg.norm(ref)
            rel = np.linalg.norm(got[s] - ref) / nrm if nrm > 0 else np.linalg.norm(got[s])
            assert rel <= BF16_STATE_REL_L2, f"{name}: slot {s} relative L2 {rel:.3e}"
        else:
            assert np.array_equal(got_bits[s], pool_bits[s]), f"{name}: untouched slot {s} changed"
