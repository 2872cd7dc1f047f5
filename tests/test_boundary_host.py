"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/ssd_scan.h declares, sizes its workspace, and rejects bad
arguments before touching the device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from mamba_ssd_chunked_varlen_gb300 import binding
from mamba_ssd_chunked_varlen_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return binding.library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ssd_scan.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(binding.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert binding.status_string(0) == "ok"
    assert "workspace" in binding.status_string(3)


def test_workspace_size(lib):
    ws = binding.ssd_scan_varlen_workspace_size
    n1 = ws(4096, 1, 16, 64, 1, 256, 256)
    # block states dominate: (ceil(T/128) + batch) blocks x H x P x N x (2 + 1/16 + 2)
    # bytes (fp16 block states with an exponent byte per 16 of them, bf16 entering
    # states; chunks longer than 128 tokens are processed as 128-token blocks)
    per_block = 16 * 64 * 256 * 4 + 16 * 64 * 256 // 16
    assert n1 >= 33 * per_block
    assert n1 < 33 * per_block + 64 * 1024
    assert ws(4096, 1, 16, 64, 1, 256, 128) == n1
    assert ws(4096, 2, 16, 64, 1, 256, 256) > n1          # more sequences, more chunks
    # with several sequences, those of at most 12 tokens hold no block and at
    # most T / 13 sequences are longer: 256 one-token sequences need
    # ceil(256/128) + 19 = 21 blocks of scratch, not ceil(256/128) + 256
    nd = ws(256, 256, 64, 64, 1, 128, 256)
    per_block_d = 64 * 64 * 128 * 4 + 64 * 64 * 128 // 16
    assert 21 * per_block_d <= nd < 21 * per_block_d + 64 * 1024
    assert ws(0, 3, 4, 32, 1, 32, 64) > 0                 # empty sequences still need a table
    assert ws(512, 1, 4, 32, 1, 512, 64) == 0             # dstate > 256 (MAX_DSTATE)
    assert ws(512, 1, 4, 32, 1, 32, 100) == 0             # unsupported chunk size
    assert ws(512, 1, 6, 32, 4, 32, 64) == 0              # nheads % ngroups != 0
    assert ws(512, 1, 4, 24, 1, 32, 64) == 0              # head_dim not a multiple of 16
    assert ws(512, 1, 4, 48, 1, 32, 64) == 0              # head_dim not a power of two
    assert ws(512, 1, 4, 256, 1, 32, 64) == 0             # head_dim > 128


def test_launch_count(lib):
    def n(T, b, H=16, P=64, G=1, N=256, Q=256):
        return binding.ssd_scan_varlen_num_launches(T, b, H, P, G, N, Q)
    assert n(4096, 1) == 3      # block states, state passing, output
    assert n(4096, 2) == 4      # + the short-sequence kernel (a batch may hold short ones)
    assert n(12, 1) == 4        # one sequence short enough for the per-token kernel
    assert n(13, 1) == 3
    assert n(0, 3) == 3         # empty sequences: no output kernel
    assert n(10, 0) == 0
    # a block-map kernel writes a block table for more than 512 sequences, or
    # when the chunk-scan grid would run more than four waves (424 blocks x 4
    # head groups here); otherwise every CTA maps its own block
    assert n(5000, 512) == 5
    assert n(5000, 513) == 5
    assert n(5000, 30) == 4     # 70 blocks x 4 head groups: under two waves
    assert n(15155, 8) == 4     # 127 blocks x 4 head groups: under four waves
    assert n(40000, 30) == 5    # 343 blocks x 4 head groups: nine waves
    # long sequences with many heads whose block states exceed the L2: block
    # states and state passing in one fused kernel (and, at 260 blocks x 32
    # head groups, the block-map kernel)
    assert n(32768, 4, 128, 64, 8, 128) == 4


def test_fused_walk_choice(lib):
    w = binding.ssd_scan_varlen_fused_walk
    assert w(32768, 4, 128, 64, 8, 128, 256)           # 4 x 8192 tokens, 128 heads
    assert w(12288, 3, 128, 64, 8, 128, 256)           # 3 x 4096 tokens
    assert not w(4096, 1, 16, 64, 1, 256, 256)         # 32 items: too few for the GPU
    assert not w(16384, 256, 64, 64, 1, 128, 256)      # short sequences
    assert w(8192, 4, 128, 64, 8, 128, 256)            # 2048 tokens each, 268 MB of states
    assert not w(16384, 8, 64, 32, 1, 64, 256)         # 2048 tokens each, 67 MB of states
    assert not w(32768, 0, 128, 64, 8, 128, 256)
    assert not w(32768, 4, 128, 64, 8, 512, 256)       # invalid sizes


def test_short_threshold(lib):
    s = binding.ssd_scan_varlen_short_threshold
    assert s(4096, 1) == 0      # one long sequence: the chunked kernels only
    assert s(12, 1) == 12 and s(13, 1) == 0
    assert s(4096, 2) == 12     # several sequences: those of <= 12 tokens
    assert s(0, 3) == 12
    assert s(10, 0) == 0
    # the launch count follows the threshold
    n = binding.ssd_scan_varlen_num_launches
    for T, b in [(4096, 1), (12, 1), (13, 1), (4096, 2), (0, 3)]:
        assert n(T, b, 16, 64, 1, 256, 256) == 2 + (T > 0) + (s(T, b) > 0)


def _call(lib, **over):
    args = dict(y=1 << 12, x=1 << 12, dt=1 << 12, A=1 << 12, B=1 << 12, C=1 << 12, D=None,
                dt_bias=None, pool=1 << 12, qsl=1 << 12, hinit=None, cidx=1 << 12,
                T=512, batch=1, H=4, P=32, G=1, N=32, slots=4, Q=64, sp=1,
                ws=1 << 12, wsb=1 << 30)
    args.update(over)
    vp = lambda v: None if v is None else ctypes.c_void_p(v)
    return lib.ssd_scan_varlen_fwd(
        vp(args["y"]), vp(args["x"]), vp(args["dt"]), vp(args["A"]), vp(args["B"]),
        vp(args["C"]), vp(args["D"]), vp(args["dt_bias"]), vp(args["pool"]), vp(args["qsl"]),
        vp(args["hinit"]), vp(args["cidx"]), args["T"], args["batch"], args["H"], args["P"],
        args["G"], args["N"], args["slots"], args["Q"], args["sp"], vp(args["ws"]),
        args["wsb"], None)


def test_host_checks_reject_before_any_launch(lib):
    # None of these reach the GPU: every one fails a host-side check first.
    assert _call(lib, x=None) == 1                 # NULL required pointer
    assert _call(lib, qsl=None) == 1
    assert _call(lib, G=3) == 1                    # nheads % ngroups
    assert _call(lib, N=512) == 2                  # dstate > MAX_DSTATE
    assert _call(lib, Q=32) == 2                   # chunk size
    assert _call(lib, P=24) == 2                   # head_dim
    assert _call(lib, x=(1 << 12) + 2) == 1        # misaligned (TMA needs 16 B)
    assert _call(lib, ws=None) == 3                # workspace
    assert _call(lib, wsb=16) == 3
    assert _call(lib, ws=(1 << 12) + 16) == 3      # workspace alignment
    assert _call(lib, T=-1) == 1
    assert _call(lib, batch=0, x=None, y=None) == 0  # empty batch: nothing to do


def _call_states(lib, **over):
    args = dict(y=1 << 12, x=1 << 12, dt=1 << 12, A=1 << 12, B=1 << 12, C=1 << 12, D=None,
                dt_bias=None, init=None, hinit=None, final=1 << 12, qsl=1 << 12,
                T=512, batch=1, H=4, P=32, G=1, N=32, Q=64, sp=1, ws=1 << 12, wsb=1 << 30)
    args.update(over)
    vp = lambda v: None if v is None else ctypes.c_void_p(v)
    return lib.ssd_scan_varlen_fwd_states(
        vp(args["y"]), vp(args["x"]), vp(args["dt"]), vp(args["A"]), vp(args["B"]),
        vp(args["C"]), vp(args["D"]), vp(args["dt_bias"]), vp(args["init"]), vp(args["hinit"]),
        vp(args["final"]), vp(args["qsl"]), args["T"], args["batch"], args["H"], args["P"],
        args["G"], args["N"], args["Q"], args["sp"], vp(args["ws"]), args["wsb"], None)


def test_states_form_host_checks(lib):
    # The separate-state-array form shares the in-place form's checks, plus its own.
    assert _call_states(lib, final=None) == 1          # final_states required
    assert _call_states(lib, final=(1 << 12) + 8) == 1  # final_states 16-byte aligned
    assert _call_states(lib, init=(1 << 12) + 4) == 1   # initial_states 16-byte aligned
    assert _call_states(lib, qsl=None) == 1
    assert _call_states(lib, N=512) == 2
    assert _call_states(lib, ws=None) == 3
    assert _call_states(lib, batch=0, final=None) == 0  # empty batch: nothing to do


def _qsl(lens):
    import numpy as np
    import torch
    return torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))


def test_host_call_plan(lib):
    """Cuts of the host-buffer call: inside (0, T), increasing, each on a
    sequence boundary or a block boundary of the sequence it falls in, at
    most the pieces asked for (0: one per 6 MiB of x, dt, B and C, 1 to 8)."""
    def plan(q, Q, n, shape=(16, 64, 1, 256)):
        return binding.ssd_scan_varlen_host_plan(q, *shape, Q, n)
    one = _qsl([4096])
    assert plan(one, 256, 1) == []
    assert plan(one, 256, 2) == [2048]
    assert plan(one, 256, 3) == [1408, 2688]          # 1365 and 2730 to the nearest 128
    assert plan(one, 256, 0) == [2048]                # 12.7 MB of inputs
    # 36.2 MB: 5 pieces, targets 819, 1638, 2457, 3276 to the nearest 128
    assert plan(one, 256, 0, (64, 64, 1, 128)) == [768, 1664, 2432, 3328]
    assert plan(_qsl([1000]), 256, 0) == []
    assert plan(one, 256, 100) == [512 * k for k in range(1, 8)]   # capped at 8 pieces
    assert plan(one, 64, 3) == [1344, 2752]           # 64-token blocks
    import numpy as np
    lens = [700, 136, 0, 900, 12, 600, 0]
    q = _qsl(lens)
    qs = q.tolist()
    for Q in (64, 128, 256):
        Qb = min(Q, 128)
        for n in range(1, 9):
            cuts = plan(q, Q, n)
            assert len(cuts) <= n - 1
            assert all(0 < c < int(q[-1]) for c in cuts)
            assert all(a < b for a, b in zip(cuts, cuts[1:]))
            for c in cuts:
                # on a sequence boundary, or a block edge of the sequence holding c
                b = int(np.searchsorted(qs, c, side="right")) - 1
                assert c in qs or (c - qs[b]) % Qb == 0, (Q, n, c)
    # 1550 falls in the second sequence: 100 + 11 blocks
    assert plan(_qsl([100, 3000]), 128, 2) == [1508]
    # 1690 rounds to 1728, past the end of its sequence: the cut is that end
    assert plan(_qsl([1600, 100, 1680]), 128, 2) == [1700]


def test_host_call_checks(lib):
    """Invalid host query_start_loc: no plan, no workspace size."""
    import torch
    bad = torch.tensor([0, 300, 200], dtype=torch.int32)
    with pytest.raises(binding.SSDError):
        binding.ssd_scan_varlen_host_plan(bad, 4, 32, 2, 64, 128, 2)
    assert binding.ssd_scan_varlen_host_workspace_size(bad, 4, 32, 2, 64, 128, 2) == 0
    ok = torch.tensor([0, 300, 500], dtype=torch.int32)
    n = binding.ssd_scan_varlen_host_workspace_size(ok, 4, 32, 2, 64, 128, 2)
    # the device copies of x, dt, B, C and y plus one scan workspace per piece
    assert n >= 500 * (2 * 4 * 32 * 2 + 4 * 2 + 2 * 2 * 64 * 2) + \
        binding.ssd_scan_varlen_workspace_size(500, 2, 4, 32, 2, 64, 128)
    assert binding.ssd_scan_varlen_host_workspace_size(ok, 4, 32, 2, 48 * 8, 128, 2) == 0
