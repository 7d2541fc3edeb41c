"""GPU parity of the backward (ssd_chunk_scan_bwd) against the fp64 backward
oracle, itself pinned by finite differences (tests/test_oracle_bwd.py).

Tolerance: max|diff| <= 1e-3 * RMS(oracle) per gradient.  The kernel sums in
fp32; the widest sums (dA, dD: one number per head over every token and
state element; ddt: P*N terms per token) gather 1e3-1e6 terms with both
signs, which puts their rounding near 1e-5 of RMS; 1e-3 keeps two orders of
margin and still fails on any wrong term."""
import numpy as np
import pytest

import oracle
from state_space_sequence_05_b300 import inputs as I

from _helpers import to_device

pytestmark = pytest.mark.gpu

TOL_BWD = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _check(wl, use_D=True, use_init=True, use_dfinal=True, seed=0):
    import torch
    from state_space_sequence_05_b300 import ssd
    fi = I.make_forward_inputs(wl)
    d = to_device(fi)
    rng = np.random.Generator(np.random.PCG64(900 + seed))
    b, T, H, P = fi.x.shape
    N = fi.B.shape[3]
    dy = rng.standard_normal((b, T, H, P)).astype(np.float32)
    dfin = rng.standard_normal((b, H, P, N)).astype(np.float32) if use_dfinal else None
    init = fi.init if use_init else None
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = ssd.ssd_chunk_scan_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"] if use_D else None,
                               t(init), t(dy), t(dfin), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.ssd_bwd(fi.x, fi.dt, fi.A, fi.B, fi.C, fi.D if use_D else None, init, dy, dfin)
    errs = {}
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit"):
        # dD is the gradient at D whether or not D was given (a missing D is 0)
        errs[k] = oracle.rel_err(g[k].cpu().numpy(), ref[k])
        assert errs[k] <= TOL_BWD, f"{k}: max|diff|/RMS = {errs[k]:.3e}"
    return errs


def test_bwd_fp32_two_groups_ragged():
    """150 steps (two stored states and a partial chunk), two batch rows, two
    groups, P 8, N 16, with D, an initial state and dL/dfinal."""
    _check(I.small_workload(batch=2, seqlen=150, nheads=4, headdim=8, dstate=16, ngroups=2,
                            chunk=64, dtype="f32", seed=61))


def test_bwd_bf16_tensor_core_shape():
    """bf16 inputs with the tensor-core layer's head shape, P 64, N 128."""
    _check(I.small_workload(batch=1, seqlen=130, nheads=2, headdim=64, dstate=128, ngroups=1,
                            chunk=128, dtype="bf16", seed=62), seed=1)


def test_bwd_bf16_mma_padded_tiles():
    """bf16 on the tensor-core gradient kernel with headdim and dstate below
    the 64 x 128 tiles (P 24, N 40: zero-padded operands), two groups of
    three heads and a ragged last chunk."""
    _check(I.small_workload(batch=2, seqlen=100, nheads=6, headdim=24, dstate=40, ngroups=2,
                            chunk=64, dtype="bf16", seed=64), seed=3)


def test_bwd_bf16_tensor_core_head_slices():
    """The tensor-core path with two batch rows and two groups of ten heads:
    each group's heads split over two gradient blocks (8 + 2), whose dB and dC
    meet in global memory; init and dL/dfinal on both state scans."""
    _check(I.small_workload(batch=2, seqlen=200, nheads=20, headdim=64, dstate=128, ngroups=2,
                            chunk=128, dtype="bf16", seed=66), seed=5)


def test_bwd_bf16_tensor_core_without_optional_inputs():
    """The tensor-core path with no D, no initial state and no dL/dfinal."""
    _check(I.small_workload(batch=1, seqlen=140, nheads=3, headdim=64, dstate=128, ngroups=1,
                            chunk=128, dtype="bf16", init="zero", seed=67),
           use_D=False, use_init=False, use_dfinal=False, seed=6)


def test_bwd_bf16_cuda_core_path():
    """bf16 with a headdim that is no multiple of 8 (P 12): the CUDA-core
    gradient kernel."""
    _check(I.small_workload(batch=1, seqlen=90, nheads=2, headdim=12, dstate=24, ngroups=1,
                            chunk=64, dtype="bf16", seed=65), seed=4)


def test_bwd_without_optional_inputs():
    _check(I.small_workload(batch=1, seqlen=64, nheads=2, headdim=4, dstate=32, ngroups=1,
                            chunk=64, dtype="f32", init="zero", seed=63),
           use_D=False, use_init=False, use_dfinal=False, seed=2)


def test_bwd_step_by_step_path():
    """headdim 128 is past the chunked path's 64: the step-by-step kernel,
    bf16 inputs, two batch rows, a ragged 64-step stretch at the end."""
    _check(I.small_workload(batch=2, seqlen=90, nheads=2, headdim=128, dstate=32, ngroups=1,
                            chunk=64, dtype="bf16", init="normal", seed=65), seed=7)


def test_bwd_no_tokens():
    """seqlen 0: dinit is dL/dfinal, every other gradient is zero."""
    _check(I.small_workload(batch=2, seqlen=0, nheads=2, headdim=64, dstate=128, ngroups=1,
                            chunk=64, dtype="bf16", init="normal", seed=66), seed=8)


def test_bwd_l8k_shape_sampled_heads():
    """The metric's layer length (b1 T8192 H80 P64 N128, bf16, init, D):
    128 chunks of the chunked backward.  The fp64 oracle walks one head at a
    time (≈0.7 s per head at 8192 steps on one host thread), so four heads
    are checked: their per-head gradients (dx, ddt, dA, dD, dinit) from the
    full 80-head call, and every gradient, dB and dC included, from a call
    on those four heads alone."""
    import torch
    from state_space_sequence_05_b300 import ssd
    fi = I.make_forward_inputs(I.WORKLOADS["l8k"])
    d = to_device(fi)
    b, T, H, P = fi.x.shape
    rng = np.random.Generator(np.random.PCG64(905))
    dy = rng.standard_normal((b, T, H, P)).astype(np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g_all = ssd.ssd_chunk_scan_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"],
                                   t(dy))
    heads = [0, 27, 53, 79]
    hsel = lambda v, ax: np.ascontiguousarray(np.take(v, heads, axis=ax))
    xs, dts, As, Ds = hsel(fi.x, 2), hsel(fi.dt, 2), fi.A[heads], fi.D[heads]
    inits, dys = hsel(fi.init, 1), hsel(dy, 2)
    # the bf16 inputs keep their exact values on the device slice
    dsl = {k: torch.index_select(d[k], 2, torch.tensor(heads, device="cuda")).contiguous()
           for k in ("x", "dt")}
    g_sub = ssd.ssd_chunk_scan_bwd(dsl["x"], dsl["dt"], t(As), d["B"], d["C"], t(Ds), t(inits),
                                   t(dys))
    torch.cuda.synchronize()
    ref = oracle.ssd_bwd(xs, dts, As, fi.B, fi.C, Ds, inits, dys, None)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit"):
        e = oracle.rel_err(g_sub[k].cpu().numpy(), ref[k])
        assert e <= TOL_BWD, f"{k} (four heads): max|diff|/RMS = {e:.3e}"
    per_head_axis = {"dx": 2, "ddt": 2, "dA": 0, "dD": 0, "dinit": 1}
    for k, ax in per_head_axis.items():
        e = oracle.rel_err(hsel(g_all[k].cpu().numpy(), ax), ref[k])
        assert e <= TOL_BWD, f"{k} (full call, sampled heads): max|diff|/RMS = {e:.3e}"
