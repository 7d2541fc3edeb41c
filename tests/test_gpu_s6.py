"""GPU parity of the Mamba-1 selective scan (a decay per channel and state)
against the fp64 oracle, through the C ABI.

The kernel computes in fp32 for both input dtypes (bf16 inputs are widened
exactly), so one tolerance serves both: max|diff| <= 1e-4 * RMS(oracle), for
y and for the final states separately.  A sequential fp32 recurrence with a
2^-22-accurate exponential keeps its error near 1e-6 of RMS; 1e-4 leaves two
orders of margin and still catches any wrong term.
"""
import numpy as np
import pytest

import oracle
from state_space_sequence_05_b300 import inputs as I

from _helpers import assert_close

pytestmark = pytest.mark.gpu

TOL_S6 = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _dev(f, device="cuda"):
    import torch
    dt = f.wl.dtype
    return {
        "x": I.as_torch(f.x, f.bits.get("x"), device, dt),
        "dt": I.as_torch(f.dt, f.bits.get("dt"), device, dt),
        "B": I.as_torch(f.B, f.bits.get("B"), device, dt),
        "C": I.as_torch(f.C, f.bits.get("C"), device, dt),
        "A": torch.from_numpy(f.A).to(device),
        "D": torch.from_numpy(f.D).to(device),
        "init": None if f.init is None else torch.from_numpy(f.init).to(device),
    }


def _run(f, use_D=True, use_init=True):
    import torch
    from state_space_sequence_05_b300 import ssd
    d = _dev(f)
    y, fin = ssd.ssd_selective_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"],
                                        d["D"] if use_D else None,
                                        d["init"] if use_init else None)
    torch.cuda.synchronize()
    return y.cpu().numpy(), fin.cpu().numpy()


def _check(f, use_D=True, use_init=True):
    y, fin = _run(f, use_D, use_init)
    yr, fr = oracle.s6_scan(f.x, f.dt, f.A, f.B, f.C, f.D if use_D else None,
                            f.init if use_init else None)
    return assert_close(y, yr, TOL_S6, "y"), assert_close(fin, fr, TOL_S6, "final")


def _wl(b, L, Dm, N, dtype, init="normal", seed=1):
    return I.S6Workload(f"s6_{b}_{L}_{Dm}_{N}", b, L, Dm, N, dtype, init, seed)


def test_s6_tiny_workload():
    """The page's usage shape family: batch 2, 128 steps, d_state 16."""
    _check(I.make_s6_inputs(I.S6_WORKLOADS["s6_tiny_fp32"]))


@pytest.mark.parametrize("N", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_s6_state_sizes_ragged(N, dtype):
    """Every supported state size; a length that is no multiple of the
    kernel's step block and a channel count that leaves idle lanes."""
    _check(I.make_s6_inputs(_wl(2, 301, 37, N, dtype, seed=40 + N)))


@pytest.mark.parametrize("L", [1, 7, 8, 15, 16, 17, 1000])
def test_s6_lengths(L):
    _check(I.make_s6_inputs(_wl(1, L, 20, 16, "bf16", seed=60 + L)))


def test_s6_without_skip_or_initial_state():
    f = I.make_s6_inputs(_wl(2, 200, 24, 64, "f32", seed=9))
    _check(f, use_D=False, use_init=False)


def test_s6_zero_length_returns_the_initial_state():
    import torch
    from state_space_sequence_05_b300 import ssd
    f = I.make_s6_inputs(_wl(2, 0, 12, 32, "f32", seed=3))
    d = _dev(f)
    y, fin = ssd.ssd_selective_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                        d["init"])
    torch.cuda.synchronize()
    assert y.shape == (2, 0, 12)
    np.testing.assert_array_equal(fin.cpu().numpy(), f.init)


def test_s6_reduces_to_ssd_on_the_gpu():
    """Shared decay per head: the selective scan on the GPU equals the SSD
    forward on the GPU (channels d = (h, p), dt and A repeated per channel)."""
    import torch
    from state_space_sequence_05_b300 import ssd
    wl = I.small_workload(batch=1, seqlen=300, nheads=4, headdim=16, dstate=32, ngroups=1,
                          chunk=64, dtype="f32", seed=77)
    fi = I.make_forward_inputs(wl)
    dev = "cuda"
    b, T, H, P, N = 1, 300, 4, 16, 32
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    ys, fs = ssd.ssd_chunk_scan_fwd(t(fi.x), t(fi.dt), t(fi.A), t(fi.B), t(fi.C), t(fi.D), 64,
                                    t(fi.init))
    y6, f6 = ssd.ssd_selective_scan_fwd(
        t(fi.x.reshape(b, T, H * P)), t(np.repeat(fi.dt, P, axis=2)),
        t(np.repeat(fi.A, P)[:, None] * np.ones((1, N), np.float32)), t(fi.B[:, :, 0]),
        t(fi.C[:, :, 0]), t(np.repeat(fi.D, P)), t(fi.init.reshape(b, H * P, N)))
    torch.cuda.synchronize()
    assert_close(y6.cpu().numpy(), ys.cpu().numpy().reshape(b, T, H * P), TOL_S6, "y")
    assert_close(f6.cpu().numpy(), fs.cpu().numpy().reshape(b, H * P, N), TOL_S6, "final")


@pytest.mark.parametrize("name", ["s6_l8k_n16", "s6_l8k_n128"])
def test_s6_full_size_sampled_channels(name):
    """The benchmarked workloads at full size, in the bench's launch
    configuration; the oracle recomputes 12 channels spread over the range."""
    f = I.make_s6_inputs(I.S6_WORKLOADS[name])
    y, fin = _run(f)
    Dm = f.wl.dmodel
    ch = np.unique(np.linspace(0, Dm - 1, 12).astype(int))
    yr, fr = oracle.s6_scan(f.x[:, :, ch], f.dt[:, :, ch], f.A[ch], f.B, f.C, f.D[ch],
                            f.init[:, ch])
    assert_close(y[:, :, ch], yr, TOL_S6, "y")
    assert_close(fin[:, ch], fr, TOL_S6, "final")


def test_s6_rejects_bad_arguments():
    import torch
    from state_space_sequence_05_b300 import ssd
    f = I.make_s6_inputs(_wl(1, 16, 8, 16, "f32", seed=5))
    d = _dev(f)
    lib = ssd.load_library()
    # dstate 24 is not supported; nothing is launched
    before = ssd.kernel_launches()
    st = lib.ssd_selective_scan_fwd(ssd._ptr(d["x"]), ssd._ptr(d["dt"]), ssd._ptr(d["A"]),
                                    ssd._ptr(d["B"]), ssd._ptr(d["C"]), None, None, 1, 16, 8, 24,
                                    ssd.SSD_DT_F32, ssd._ptr(torch.empty(1, 16, 8, device="cuda")),
                                    None, None)
    assert st == ssd.SSD_ERR_UNSUPPORTED
    st = lib.ssd_selective_scan_fwd(None, ssd._ptr(d["dt"]), ssd._ptr(d["A"]), ssd._ptr(d["B"]),
                                    ssd._ptr(d["C"]), None, None, 1, 16, 8, 16, ssd.SSD_DT_F32,
                                    ssd._ptr(torch.empty(1, 16, 8, device="cuda")), None, None)
    assert st == ssd.SSD_ERR_INVALID
    assert ssd.kernel_launches() == before
