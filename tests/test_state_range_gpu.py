"""Block states cross the workspace as fp16 scaled by a power of two per
group of 16 values.  These cases drive the states far from the magnitudes of
the standard workloads (x and B scaled up or down by 2^12 and more, so that
plain fp16 would overflow or lose every value to underflow) and check that
y and the final states still match the oracle at the usual tolerances."""
from __future__ import annotations

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


def _scaled(w, sx: float, sb: float, spool: float):
    """The workload with x, B and the pool scaled by powers of two (exact in
    bf16 / fp32), so the oracle sees exactly the scaled values."""
    xf = W.bf16_bits_to_f32(w.x) * np.float32(sx)
    bf = W.bf16_bits_to_f32(w.B) * np.float32(sb)
    w.x = W.f32_to_bf16_bits(xf)
    w.B = W.f32_to_bf16_bits(bf)
    w.ssm_pool = (w.ssm_pool * np.float32(spool)).astype(np.float32)
    return w


@pytest.mark.parametrize("sx,sb,spool", [
    (2.0 ** 12, 2.0 ** 10, 2.0 ** 20),     # states ~2^22: plain fp16 overflows
    (2.0 ** -12, 2.0 ** -10, 2.0 ** -20),  # states ~2^-22: plain fp16 flushes them
    (2.0 ** 14, 2.0 ** -14, 1.0),          # large x, tiny B
])
def test_state_magnitudes(sx, sb, spool):
    w = W.make_workload("range", [700, 300, 129, 1000], 8, 64, 2, 128, 256, max_slots=6,
                        seed=61, has_init_p=0.75)
    w = _scaled(w, sx, sb, spool)
    y, pool, _, ws = run_cuda(w)
    import mamba_ssd_chunked_varlen_gb300 as pkg
    assert pkg.ssd_scan_varlen_read_errors(ws) == 0
    y_ref, pool_ref = recurrence.run_workload(w)
    check_y(y_to_f64(y), y_ref, what=f"x*{sx} B*{sb} pool*{spool}")
    check_slots(pool.cpu().numpy(), pool_ref, w.ssm_pool, w, what=f"x*{sx} B*{sb} pool*{spool}")
