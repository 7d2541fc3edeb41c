"""GPU side of context parallelism: the two device steps against fp64, and
the whole scheme run in one process over slices of a sequence (the slices
are processed one after another; only the exchange of a multi-GPU run is
replaced by a list).  Tolerances: the sums and compositions in fp32, 1e-5
relative; the forward outputs, the bf16-input bar 1e-2 * RMS."""
import numpy as np
import pytest

import oracle
from state_space_sequence_05_b300 import inputs as I

from _helpers import TOL, assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_segment_decay(dtype):
    import torch
    from state_space_sequence_05_b300 import ssd
    wl = I.small_workload(batch=3, seqlen=1000, nheads=5, headdim=8, dstate=16, ngroups=1,
                          chunk=64, dtype=dtype, seed=51)
    fi = I.make_forward_inputs(wl)
    d = to_device(fi)
    a = ssd.ssd_segment_decay(d["dt"], d["A"])
    torch.cuda.synchronize()
    want = fi.dt.astype(np.float64).sum(axis=1) * fi.A.astype(np.float64)[None, :]
    assert np.max(np.abs(a.cpu().numpy() - want) / np.abs(want)) < 1e-5


def test_segment_combine():
    import torch
    from state_space_sequence_05_b300 import ssd
    rng = np.random.Generator(np.random.PCG64(52))
    R, b, H, P, N = 4, 2, 3, 8, 16
    a = -rng.uniform(0.0, 3.0, (R, b, H)).astype(np.float32)
    S = rng.standard_normal((R, b, H, P, N)).astype(np.float32)
    h0 = rng.standard_normal((b, H, P, N)).astype(np.float32)
    t = lambda v: torch.from_numpy(v).cuda()
    for init in (h0, None):
        out = ssd.ssd_segment_combine(t(a), t(S), None if init is None else t(init))
        torch.cuda.synchronize()
        want = np.zeros((R + 1, b, H, P, N))
        if init is not None:
            want[0] = init
        for r in range(R):
            want[r + 1] = np.exp(a[r].astype(np.float64))[:, :, None, None] * want[r] + S[r]
        assert oracle.rel_err(out.cpu().numpy(), want) < 1e-5


def _cp_emulated(d, bounds, states_only):
    """The context-parallel scheme on one GPU, one slice after the other:
    each slice's end state from a zero state (the states-only pass, or a
    forward whose y is dropped), the exchange as a list, the composition
    kernel, each slice's forward from its entering state."""
    import torch
    from state_space_sequence_05_b300 import ssd
    R = len(bounds) - 1
    sl = lambda v, r: v[:, bounds[r]:bounds[r + 1]].contiguous()
    S, a = [], []
    for r in range(R):
        if states_only:
            s = ssd.ssd_chunk_scan_states(sl(d["x"], r), sl(d["dt"], r), d["A"], sl(d["B"], r), 256)
        else:
            _, s = ssd.ssd_chunk_scan_fwd(sl(d["x"], r), sl(d["dt"], r), d["A"], sl(d["B"], r),
                                          sl(d["C"], r), None, 256, None)
        S.append(s)
        a.append(ssd.ssd_segment_decay(sl(d["dt"], r), d["A"]))
    h_in = ssd.ssd_segment_combine(torch.stack(a).contiguous(), torch.stack(S).contiguous(),
                                   d["init"])
    ys, fins = [], []
    for r in range(R):
        y, f = ssd.ssd_chunk_scan_fwd(sl(d["x"], r), sl(d["dt"], r), d["A"], sl(d["B"], r),
                                      sl(d["C"], r), d["D"], 256, h_in[r].contiguous())
        ys.append(y)
        fins.append(f)
    return torch.cat(ys, dim=1), fins[-1], h_in


def test_context_parallel_slices_on_one_gpu():
    """A b2 T1100 layer on the tensor-core path cut into slices of 256, 500
    and 344 tokens, with the states-only first pass and with a forward in its
    place: the concatenated y and the last final state against the oracle
    and the unsplit forward."""
    import torch
    from state_space_sequence_05_b300 import ssd
    wl = I.small_workload(batch=2, seqlen=1100, nheads=4, ngroups=2, chunk=256, seed=53)
    fi = I.make_forward_inputs(wl)
    d = to_device(fi)
    bounds = (0, 256, 756, 1100)
    y_ref, fin_ref = oracle.ssd_scan(fi.x, fi.dt, fi.A, fi.B, fi.C, fi.D, fi.init)
    y_whole, _ = ssd.ssd_chunk_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 256,
                                        d["init"])
    for states_only in (True, False):
        y, fin, h_in = _cp_emulated(d, bounds, states_only)
        torch.cuda.synchronize()
        y = y.cpu().numpy()
        assert_close(y, y_ref, TOL["bf16"], "y")
        assert_close(fin.cpu().numpy(), fin_ref, TOL["bf16"], "final")
        assert_close(h_in[3].cpu().numpy(), fin_ref, TOL["bf16"], "composed end state")
        assert_close(y, y_whole.cpu().numpy(), TOL["bf16"], "y against the unsplit forward")


def test_context_parallel_first_pass_timed():
    """The 2.7B-shaped layer (b1 T8192 H80) in two slices of 4096 tokens:
    the per-slice first pass timed as a states-only pass and as a forward
    (CUDA events, median of 7 after 2 warm-ups), results equal."""
    import torch
    from state_space_sequence_05_b300 import ssd
    fi = I.make_forward_inputs(I.WORKLOADS["l8k"])
    d = to_device(fi)
    x, dt, B, C = (d[k][:, :4096].contiguous() for k in ("x", "dt", "B", "C"))

    def timed(fn):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(7):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1000)
        return sorted(ts)[3]

    t_states = timed(lambda: ssd.ssd_chunk_scan_states(x, dt, d["A"], B, 256))
    t_fwd = timed(lambda: ssd.ssd_chunk_scan_fwd(x, dt, d["A"], B, C, None, 256, None))
    s1 = ssd.ssd_chunk_scan_states(x, dt, d["A"], B, 256)
    _, s2 = ssd.ssd_chunk_scan_fwd(x, dt, d["A"], B, C, None, 256, None)
    torch.cuda.synchronize()
    assert_close(s1.cpu().numpy(), s2.cpu().numpy(), TOL["bf16"], "end state")
    print(f"first pass per 4096-token slice: states-only {t_states:.1f} us, "
          f"forward {t_fwd:.1f} us")
