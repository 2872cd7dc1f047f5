"""Seeded synthetic inputs for the Mamba-2 SSD varlen forward prefill scan.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds input generation only (random draws, bf16 storage
rounding, the five workload shapes); none of the scan's own arithmetic lives
here.

Shapes and dtypes follow the "Tensor shapes" section of the Modular page
"Mamba2SSDChunkScanVarlenFwdInplace":

    x, y      (total_len, nheads, head_dim)            bf16
    dt        (total_len, nheads)                      bf16
    A         (nheads,)                                fp32
    B, C      (total_len, ngroups, dstate)             bf16
    D         (nheads,)  optional                      fp32
    dt_bias   (nheads,)  optional                      fp32
    ssm_pool  (max_slots, nheads, head_dim, dstate)    fp32, updated in place
    query_start_loc (batch + 1,)                       int32
    has_initial_state (batch,) optional                bool (uint8 here)
    cache_indices (batch,)                             uint32

bf16 tensors are carried as uint16 bit patterns so that NumPy (which has no
bfloat16 type) and the C oracle see exactly the bits the GPU sees.

Value recipe (the same for every workload; the pages print no data):
    x, B, C        ~ N(0, 1), rounded to bf16 (round to nearest even)
    dt (raw)       ~ N(0, 0.5), rounded to bf16
    dt_bias        = log(expm1(u)), u = exp(U[ln 1e-3, ln 1e-1])  (so that
                     softplus(dt_bias) is log-uniform in [1e-3, 1e-1])
    (dt_softplus off: dt = 0.2 |N(0, 0.5)| and dt_bias = u, steps that are
     already positive, as a caller that skips softplus would pass)
    A              = -exp(U[ln 1, ln 16])
    D              ~ N(0, 1)
    ssm_pool       ~ N(0, 0.1), fp32
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even).

    Returns the uint16 bit patterns.  Inputs here are finite, so NaN handling
    is not needed.  Works through the array in pieces of 4 Mi elements with
    in-place integer steps (the large workloads hold ~10^8 values).
    """
    src = np.ascontiguousarray(a, dtype=np.float32)
    u = src.view(np.uint32).reshape(-1)
    out = np.empty(u.shape, dtype=np.uint16)
    step = 1 << 22
    for s in range(0, u.shape[0], step):
        v = u[s:s + step]
        t = v >> np.uint32(16)
        t &= np.uint32(1)          # the lowest kept bit: ties go to even
        t += v
        t += np.uint32(0x7FFF)
        t >>= np.uint32(16)
        out[s:s + step] = t
    return out.reshape(src.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen uint16 bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Workload:
    """One problem instance: sizes plus the arrays of every op argument."""

    name: str
    nheads: int
    head_dim: int
    ngroups: int
    dstate: int
    chunk_size: int
    x: np.ndarray            # uint16 (T, H, P)
    dt: np.ndarray           # uint16 (T, H)
    A: np.ndarray            # float32 (H,)
    B: np.ndarray            # uint16 (T, G, N)
    C: np.ndarray            # uint16 (T, G, N)
    D: Optional[np.ndarray]  # float32 (H,) or None
    dt_bias: Optional[np.ndarray]  # float32 (H,) or None
    ssm_pool: np.ndarray     # float32 (max_slots, H, P, N)
    query_start_loc: np.ndarray   # int32 (batch + 1,)
    has_initial_state: Optional[np.ndarray]  # uint8 (batch,) or None
    cache_indices: np.ndarray     # uint32 (batch,)
    dt_softplus: bool = True

    @property
    def total_len(self) -> int:
        return int(self.x.shape[0])

    @property
    def batch(self) -> int:
        return int(self.query_start_loc.shape[0] - 1)

    @property
    def max_slots(self) -> int:
        return int(self.ssm_pool.shape[0])

    @property
    def seq_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc.astype(np.int64))

    def dims(self) -> dict:
        return dict(total_len=self.total_len, batch=self.batch, nheads=self.nheads,
                    head_dim=self.head_dim, ngroups=self.ngroups, dstate=self.dstate,
                    max_slots=self.max_slots, chunk_size=self.chunk_size)


def make_workload(name: str, seq_lens, nheads: int, head_dim: int, ngroups: int,
                  dstate: int, chunk_size: int, max_slots: int, seed: int,
                  has_init_p: float = 0.0, cache_indices=None,
                  with_D: bool = True, with_dt_bias: bool = True,
                  dt_softplus: bool = True) -> Workload:
    """Draw one workload with the value recipe in the module docstring.

    Draw order is fixed (lengths are given by the caller): x, dt, B, C, A,
    dt_bias, D, pool, cache indices, has_initial_state.
    """
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    batch = int(seq_lens.shape[0])
    T = int(seq_lens.sum())
    H, P, G, N = nheads, head_dim, ngroups, dstate
    qsl = np.zeros(batch + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(seq_lens)

    x = f32_to_bf16_bits(rng.standard_normal((T, H, P), dtype=np.float32))
    dt_raw = rng.standard_normal((T, H), dtype=np.float32) * np.float32(0.5)
    if not dt_softplus:
        # Without softplus the op uses dt + dt_bias as the step directly, so a
        # caller passes steps that are already positive.
        dt_raw = np.abs(dt_raw) * np.float32(0.2)
    dt = f32_to_bf16_bits(dt_raw)
    B = f32_to_bf16_bits(rng.standard_normal((T, G, N), dtype=np.float32))
    C = f32_to_bf16_bits(rng.standard_normal((T, G, N), dtype=np.float32))
    A = (-np.exp(rng.uniform(np.log(1.0), np.log(16.0), H))).astype(np.float32)
    u = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), H))
    dt_bias = (np.log(np.expm1(u)) if dt_softplus else u).astype(np.float32)
    D = rng.standard_normal(H).astype(np.float32)
    pool = (rng.standard_normal((max_slots, H, P, N), dtype=np.float32) * np.float32(0.1))
    if cache_indices is None:
        cache_indices = rng.permutation(max_slots)[:batch]
    cache_indices = np.asarray(cache_indices, dtype=np.uint32)
    if has_init_p > 0.0:
        has_init = (rng.random(batch) < has_init_p).astype(np.uint8)
    else:
        has_init = np.zeros(batch, dtype=np.uint8)
    return Workload(name=name, nheads=H, head_dim=P, ngroups=G, dstate=N,
                    chunk_size=chunk_size, x=x, dt=dt, A=A, B=B, C=C,
                    D=D if with_D else None,
                    dt_bias=dt_bias if with_dt_bias else None,
                    ssm_pool=pool, query_start_loc=qsl,
                    has_initial_state=has_init, cache_indices=cache_indices,
                    dt_softplus=dt_softplus)


def _ragged_lengths(rng: np.random.Generator, n: int, lo: int, hi: int, avoid_multiple: int):
    out = []
    while len(out) < n:
        v = int(rng.integers(lo, hi + 1))
        if v % avoid_multiple == 0:
            continue
        out.append(v)
    return out


# Workload names, in the order they are listed for this op.
WORKLOADS = ("tiny", "kernelindex", "ragged", "nemotron_h", "serving_mix", "decode",
             "nemotron_h_2k")


def workload(name: str, seed: Optional[int] = None) -> Workload:
    """The standard workloads.

    tiny          1 x 512 tokens, H=4, P=32, G=1, N=32, chunk 64, no initial state.
    kernelindex   1 x 4096 tokens, H=16, P=64, G=1, N=256, chunk 256: the head and
                  state shape of the kernelindex "Mamba chunk scan with segsum"
                  workload (its 16 cases are not published), no initial state.
    ragged        8 sequences, lengths U[1, 4096] (never a multiple of 256),
                  H=16, P=64, G=1, N=256, chunk 256, 64-slot pool, initial state
                  with p = 0.5.
    nemotron_h    4 x 8192 tokens, H=128, P=64, G=8, N=128, chunk 256, 16-slot
                  pool, every sequence with an initial state.
    serving_mix   256 sequences, geometric lengths with mean 64, H=64, P=64, G=1,
                  N=128, chunk 256, 512-slot pool, initial state with p = 0.8.
    decode        256 sequences of 1 token each (a decode step of the serving
                  shape: H=64, P=64, G=1, N=128, chunk 256, 512-slot pool), every
                  sequence with an initial state: the pool read-modify-write case.
    nemotron_h_2k nemotron_h with 4 x 2048 tokens: the smallest call of that
                  shape whose chunk states exceed the L2 (so it takes the fused
                  walk), ~1 GB on the device, for profiling the walk.

    For tiny and kernelindex the pool has 4 slots and one random slot is
    written, so that the untouched-slot check has something to check.
    """
    sp = workload_spec(name, seed)
    return make_workload(name, sp["lens"], sp["nheads"], sp["head_dim"], sp["ngroups"],
                         sp["dstate"], sp["chunk_size"], max_slots=sp["max_slots"],
                         seed=sp["seed"], has_init_p=sp["has_init_p"])


def workload_spec(name: str, seed: Optional[int] = None) -> dict:
    """Sizes, sequence lengths, pool size, seed and initial-state probability
    of a standard workload (see `workload`), without drawing its arrays."""
    idx = WORKLOADS.index(name)
    seed = idx if seed is None else seed

    def spec(lens, H, P, G, N, Q, max_slots, has_init_p=0.0):
        return dict(lens=[int(v) for v in lens], nheads=H, head_dim=P, ngroups=G, dstate=N,
                    chunk_size=Q, max_slots=max_slots, seed=seed, has_init_p=has_init_p)

    if name == "tiny":
        return spec([512], 4, 32, 1, 32, 64, 4)
    if name == "kernelindex":
        return spec([4096], 16, 64, 1, 256, 256, 4)
    if name == "ragged":
        lens = _ragged_lengths(np.random.default_rng([seed, 1]), 8, 1, 4096, 256)
        return spec(lens, 16, 64, 1, 256, 256, 64, 0.5)
    if name == "nemotron_h":
        return spec([8192] * 4, 128, 64, 8, 128, 256, 16, 1.0)
    if name == "serving_mix":
        lens = np.random.default_rng([seed, 1]).geometric(1.0 / 64.0, 256)
        return spec(lens, 64, 64, 1, 128, 256, 512, 0.8)
    if name == "nemotron_h_2k":
        return spec([2048] * 4, 128, 64, 8, 128, 256, 16, 1.0)
    if name == "decode":
        return spec([1] * 256, 64, 64, 1, 128, 256, 512, 1.0)
    raise KeyError(name)


@dataclasses.dataclass
class DeviceWorkload:
    """A workload drawn directly on a CUDA device (for timing large workloads
    without a host round trip): the sizes and small host arrays of `Workload`
    plus the device tensors in `dev` (x, dt, A, B, C, D, dt_bias, pool, qsl,
    hinit, cidx).  Same value recipe as `make_workload`, drawn by torch's
    seeded device generator instead of NumPy, so the values differ from the
    host workload of the same name."""

    name: str
    nheads: int
    head_dim: int
    ngroups: int
    dstate: int
    chunk_size: int
    query_start_loc: np.ndarray
    has_initial_state: np.ndarray
    cache_indices: np.ndarray
    dev: dict
    dt_softplus: bool = True

    @property
    def total_len(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def batch(self) -> int:
        return int(self.query_start_loc.shape[0] - 1)

    @property
    def seq_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc.astype(np.int64))


def device_workload(name: str, device, seed: Optional[int] = None) -> DeviceWorkload:
    """The standard workload `name` drawn on `device` (see DeviceWorkload)."""
    import torch

    sp = workload_spec(name, seed)
    H, P, G, N = sp["nheads"], sp["head_dim"], sp["ngroups"], sp["dstate"]
    lens = np.asarray(sp["lens"], dtype=np.int64)
    batch = int(lens.shape[0])
    T = int(lens.sum())
    qsl = np.zeros(batch + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(lens)
    rng = np.random.default_rng([sp["seed"], 11])
    A = (-np.exp(rng.uniform(np.log(1.0), np.log(16.0), H))).astype(np.float32)
    u = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), H))
    dt_bias = np.log(np.expm1(u)).astype(np.float32)
    D = rng.standard_normal(H).astype(np.float32)
    cidx = rng.permutation(sp["max_slots"])[:batch].astype(np.uint32)
    hinit = ((rng.random(batch) < sp["has_init_p"]) if sp["has_init_p"] > 0.0
             else np.zeros(batch, bool)).astype(np.uint8)
    g = torch.Generator(device=device)
    g.manual_seed(int(sp["seed"]) * 7919 + 17)

    def normal(shape, std=1.0):
        return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std)

    dev = dict(
        x=normal((T, H, P)).to(torch.bfloat16),
        dt=normal((T, H), 0.5).to(torch.bfloat16),
        B=normal((T, G, N)).to(torch.bfloat16),
        C=normal((T, G, N)).to(torch.bfloat16),
        pool=normal((sp["max_slots"], H, P, N), 0.1),
        A=torch.from_numpy(A).to(device), D=torch.from_numpy(D).to(device),
        dt_bias=torch.from_numpy(dt_bias).to(device),
        qsl=torch.from_numpy(qsl).to(device), hinit=torch.from_numpy(hinit).to(device),
        cidx=torch.from_numpy(cidx.astype(np.int32)).to(device))
    return DeviceWorkload(name=name, nheads=H, head_dim=P, ngroups=G, dstate=N,
                          chunk_size=sp["chunk_size"], query_start_loc=qsl,
                          has_initial_state=hinit, cache_indices=cidx, dev=dev)


def random_small_workload(seed: int, max_total: int = 600) -> Workload:
    """A random small problem (fuzzing): random batch, lengths (including 0 and
    1), head/group/state sizes from the supported sets and random optionals."""
    rng = np.random.default_rng([seed, 7])
    P = int(rng.choice([32, 64, 128]))
    N = int(rng.choice([32, 64, 128, 256]))
    G = int(rng.choice([1, 2]))
    H = G * int(rng.choice([1, 2, 3]))
    Q = int(rng.choice([64, 128, 256]))
    batch = int(rng.integers(1, 6))
    lens = rng.integers(0, max(2, max_total // batch), batch)
    if rng.random() < 0.3:
        lens[rng.integers(0, batch)] = 1
    max_slots = batch + int(rng.integers(0, 4))
    return make_workload(f"fuzz{seed}", lens, H, P, G, N, Q, max_slots=max_slots,
                         seed=seed + 1000, has_init_p=0.5,
                         with_D=bool(rng.random() < 0.8),
                         with_dt_bias=bool(rng.random() < 0.8),
                         dt_softplus=bool(rng.random() < 0.85))
