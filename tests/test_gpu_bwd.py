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
    g = ssd.ssd_chunk_scan_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"] if use_D else None,
                               t(init), t(dy), t(dfin))
    torch.cuda.synchronize()
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


def test_bwd_without_optional_inputs():
    _check(I.small_workload(batch=1, seqlen=64, nheads=2, headdim=4, dstate=32, ngroups=1,
                            chunk=64, dtype="f32", init="zero", seed=63),
           use_D=False, use_init=False, use_dfinal=False, seed=2)
