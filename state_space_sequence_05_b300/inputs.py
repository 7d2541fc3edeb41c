"""Seeded synthetic inputs for the SSD layer forward and the decode step.

This module draws and rounds random numbers and nothing else: it holds none
of the layer's arithmetic.  Tests feed the same arrays to the fp64 oracle and
to the CUDA library, and the bench uses it to build its workloads.

Value distributions (the workload recipe):

* x, B, C ~ N(0, 1); D ~ N(0, 1), one scalar per head.
* A_h = -exp(U(ln 1, ln 16)), one scalar per head.
* dt = softplus(N(0, 0.5^2) + b_h) with a per-head bias b_h = softplus^-1(u_h)
  and u_h log-uniform on [1e-3, 1e-1]: the bias sets the centre of each
  head's step size; individual values spread around it (no clamp).  softplus
  is how a Mamba block makes dt positive ("20.1 상태 공간 모델 (SSM)", sec. 2);
  here it only shapes the synthetic dt, the layer takes dt as given.
* initial state: zero, or N(0, 0.1^2) elementwise.
* varlen: sequence lengths floor(exp(U(ln 64, ln 8192))), packed back to back.

bf16 workloads round x, dt, B and C to bf16 on the host (round to nearest,
ties to even) before either side sees them; both the oracle and the GPU read
the rounded values.  A, D and the initial state stay fp32.

Draw order from ``numpy.random.Generator(PCG64(seed))``: (varlen lengths),
x, dt noise, B, C, A, D, dt bias u_h, initial state.

The Mamba-1 selective scan (a decay per channel d and state n) uses the same
recipe per channel instead of per head, except A[d, n] = -exp(A_log) with
A_log ~ N(0, 1) elementwise, the parameterisation of the selective-SSM
example in "20.1 상태 공간 모델 (SSM)", sec. 5.  Draw order: x, dt noise, B,
C, A_log, D, dt bias u_d, initial state.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np


@dataclass(frozen=True)
class Workload:
    """Shape and dtype of one SSD forward problem."""
    name: str
    batch: int
    seqlen: int            # tokens per row; total packed tokens for varlen
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str             # "f32" or "bf16": dtype of x, dt, B, C
    init: str              # "zero" or "normal"
    nseq: int = 0          # > 0: varlen, `nseq` packed sequences (batch 1)
    seed: int = 1000


# Named workloads.  seqlen of the varlen workload is filled in from the drawn
# lengths (see make_forward_inputs).
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 256, 2, 16, 16, 1, 64, "f32", "zero", seed=1000),
    "l2k_b4": Workload("l2k_b4", 4, 2048, 80, 64, 128, 1, 256, "bf16", "zero", seed=1001),
    "l8k": Workload("l8k", 1, 8192, 80, 64, 128, 1, 256, "bf16", "normal", seed=1002),
    "l64k": Workload("l64k", 1, 65536, 80, 64, 128, 1, 256, "bf16", "normal", seed=1002),
    "varlen64": Workload("varlen64", 1, 0, 64, 64, 128, 8, 256, "bf16", "zero", nseq=64, seed=1003),
}


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    steps: int
    dtype: str = "bf16"
    seed: int = 1004


DECODE_WORKLOADS = {
    "decode_b256": DecodeWorkload("decode_b256", 256, 80, 64, 128, 1, 128),
}


def bf16_round(a: np.ndarray):
    """Round float32 values to bf16, ties to even.

    Returns ``(bits, values)``: the uint16 bf16 bit patterns and the same
    numbers as exact float32 values.  Inputs must be finite.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    bits = (u >> 16).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    return bits, vals


def _softplus(z):
    z = np.asarray(z, dtype=np.float64)
    return np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))


def _softplus_inv(u):
    u = np.asarray(u, dtype=np.float64)
    return np.log(np.expm1(u))


def varlen_lengths(rng: np.random.Generator, nseq: int, lo: int = 64, hi: int = 8192):
    return np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi), nseq))).astype(np.int64)


@dataclass
class ForwardInputs:
    """One forward problem.  Arrays are float32 (values exactly representable
    in ``dtype``); ``bits`` holds the bf16 bit patterns for bf16 workloads."""
    wl: Workload
    x: np.ndarray          # [b, T, H, P]
    dt: np.ndarray         # [b, T, H]
    A: np.ndarray          # [H]
    B: np.ndarray          # [b, T, G, N]
    C: np.ndarray          # [b, T, G, N]
    D: np.ndarray          # [H]
    init: Optional[np.ndarray]        # [nseq or b, H, P, N] or None
    cu_seqlens: Optional[np.ndarray]  # int32 [nseq + 1] or None
    bits: dict = field(default_factory=dict)

    @property
    def nseq(self):
        return self.wl.batch if self.cu_seqlens is None else len(self.cu_seqlens) - 1


def make_forward_inputs(wl: Workload, seed: Optional[int] = None,
                        init_zero_as_none: bool = True) -> ForwardInputs:
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    cu = None
    if wl.nseq > 0:
        lens = varlen_lengths(rng, wl.nseq)
        cu = np.zeros(wl.nseq + 1, np.int32)
        cu[1:] = np.cumsum(lens)
        wl = replace(wl, batch=1, seqlen=int(cu[-1]))
    b, T, H, P, N, G = wl.batch, wl.seqlen, wl.nheads, wl.headdim, wl.dstate, wl.ngroups
    x = rng.standard_normal((b, T, H, P), dtype=np.float32)
    noise = rng.standard_normal((b, T, H), dtype=np.float32) * np.float32(0.5)
    Bm = rng.standard_normal((b, T, G, N), dtype=np.float32)
    Cm = rng.standard_normal((b, T, G, N), dtype=np.float32)
    A = (-np.exp(rng.uniform(np.log(1.0), np.log(16.0), H))).astype(np.float32)
    D = rng.standard_normal(H).astype(np.float32)
    u = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), H))
    dt = _softplus(noise.astype(np.float64) + _softplus_inv(u)[None, None, :]).astype(np.float32)
    nseq = b if cu is None else wl.nseq
    if wl.init == "normal":
        init = (rng.standard_normal((nseq, H, P, N), dtype=np.float32) * np.float32(0.1))
    else:
        init = None if init_zero_as_none else np.zeros((nseq, H, P, N), np.float32)
    bits = {}
    if wl.dtype == "bf16":
        for name in ("x", "dt", "B", "C"):
            arr = {"x": x, "dt": dt, "B": Bm, "C": Cm}[name]
            bits[name], vals = bf16_round(arr)
            if name == "x":
                x = vals
            elif name == "dt":
                dt = vals
            elif name == "B":
                Bm = vals
            else:
                Cm = vals
    elif wl.dtype != "f32":
        raise ValueError(f"unknown dtype {wl.dtype}")
    return ForwardInputs(wl, x, dt, A, Bm, Cm, D, init, cu, bits)


@dataclass
class DecodeInputs:
    wl: DecodeWorkload
    state0: np.ndarray     # [b, H, P, N] float32
    A: np.ndarray          # [H]
    D: np.ndarray          # [H]
    dt_bias_u: np.ndarray  # [H] centre of each head's dt


@dataclass
class DecodeToken:
    x: np.ndarray          # [b, H, P]
    dt: np.ndarray         # [b, H]
    B: np.ndarray          # [b, G, N]
    C: np.ndarray          # [b, G, N]
    bits: dict = field(default_factory=dict)


def make_decode_inputs(wl: DecodeWorkload) -> DecodeInputs:
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    b, H, P, N = wl.batch, wl.nheads, wl.headdim, wl.dstate
    A = (-np.exp(rng.uniform(np.log(1.0), np.log(16.0), H))).astype(np.float32)
    D = rng.standard_normal(H).astype(np.float32)
    u = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), H))
    state0 = rng.standard_normal((b, H, P, N), dtype=np.float32) * np.float32(0.1)
    return DecodeInputs(wl, state0, A, D, u)


def make_decode_token(wl: DecodeWorkload, dec: DecodeInputs, step: int) -> DecodeToken:
    """Token `step` of the decode run, from its own stream PCG64([seed, step])."""
    rng = np.random.Generator(np.random.PCG64([wl.seed, step]))
    b, H, P, N, G = wl.batch, wl.nheads, wl.headdim, wl.dstate, wl.ngroups
    x = rng.standard_normal((b, H, P), dtype=np.float32)
    noise = rng.standard_normal((b, H), dtype=np.float32) * np.float32(0.5)
    Bm = rng.standard_normal((b, G, N), dtype=np.float32)
    Cm = rng.standard_normal((b, G, N), dtype=np.float32)
    dt = _softplus(noise.astype(np.float64) + _softplus_inv(dec.dt_bias_u)[None, :]).astype(np.float32)
    bits = {}
    if wl.dtype == "bf16":
        bits["x"], x = bf16_round(x)
        bits["dt"], dt = bf16_round(dt)
        bits["B"], Bm = bf16_round(Bm)
        bits["C"], Cm = bf16_round(Cm)
    return DecodeToken(x, dt, Bm, Cm, bits)


def small_workload(name="small", batch=2, seqlen=300, nheads=4, headdim=64, dstate=128,
                   ngroups=2, chunk=128, dtype="bf16", init="normal", nseq=0, seed=7):
    """Convenience constructor for test-sized problems."""
    return Workload(name, batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype,
                    init, nseq, seed)


def as_torch(arr_f32: np.ndarray, bits: Optional[np.ndarray], device, dtype: str):
    """Move one input to `device` as fp32, or as bf16 from its bit patterns."""
    import torch
    if dtype == "bf16":
        assert bits is not None
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr_f32, dtype=np.float32))
    return t.to(device)


@dataclass(frozen=True)
class S6Workload:
    """Shape and dtype of one selective-scan problem."""
    name: str
    batch: int
    seqlen: int
    dmodel: int
    dstate: int
    dtype: str             # "f32" or "bf16": dtype of x, dt, B, C
    init: str              # "zero" or "normal"
    seed: int = 1010


# The long workloads have the token count and channel count (80 heads x 64)
# of the SSD layer workload, with Mamba-1's usual state size and with SSD's.
S6_WORKLOADS = {
    "s6_tiny_fp32": S6Workload("s6_tiny_fp32", 2, 128, 64, 16, "f32", "normal", 1010),
    "s6_l8k_n16": S6Workload("s6_l8k_n16", 1, 8192, 5120, 16, "bf16", "normal", 1011),
    "s6_l8k_n128": S6Workload("s6_l8k_n128", 1, 8192, 5120, 128, "bf16", "normal", 1012),
}


@dataclass
class S6Inputs:
    wl: S6Workload
    x: np.ndarray          # [b, L, Dm]
    dt: np.ndarray         # [b, L, Dm]
    A: np.ndarray          # [Dm, N]
    B: np.ndarray          # [b, L, N]
    C: np.ndarray          # [b, L, N]
    D: np.ndarray          # [Dm]
    init: Optional[np.ndarray]   # [b, Dm, N] or None
    bits: dict = field(default_factory=dict)


def make_s6_inputs(wl: S6Workload, seed: Optional[int] = None) -> S6Inputs:
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    b, L, Dm, N = wl.batch, wl.seqlen, wl.dmodel, wl.dstate
    x = rng.standard_normal((b, L, Dm), dtype=np.float32)
    noise = rng.standard_normal((b, L, Dm), dtype=np.float32) * np.float32(0.5)
    Bm = rng.standard_normal((b, L, N), dtype=np.float32)
    Cm = rng.standard_normal((b, L, N), dtype=np.float32)
    A = (-np.exp(rng.standard_normal((Dm, N)))).astype(np.float32)
    D = rng.standard_normal(Dm).astype(np.float32)
    u = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), Dm))
    dt = _softplus(noise.astype(np.float64) + _softplus_inv(u)[None, None, :]).astype(np.float32)
    init = (rng.standard_normal((b, Dm, N), dtype=np.float32) * np.float32(0.1)
            if wl.init == "normal" else None)
    bits = {}
    if wl.dtype == "bf16":
        bits["x"], x = bf16_round(x)
        bits["dt"], dt = bf16_round(dt)
        bits["B"], Bm = bf16_round(Bm)
        bits["C"], Cm = bf16_round(Cm)
    elif wl.dtype != "f32":
        raise ValueError(f"unknown dtype {wl.dtype}")
    return S6Inputs(wl, x, dt, A, Bm, Cm, D, init, bits)
