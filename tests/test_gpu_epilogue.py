"""GPU parity of the fused epilogue options of ssd_chunk_scan_fwd_ex (the
tensor-core kernel's epilogue variant): dt = softplus(dt + dt_bias) in the
decay tables, y *= silu(z), bf16 y.  The oracle side applies the same steps
in fp64 around the sequential recurrence (oracle.softplus before it,
oracle.silu_gate after it).  Tolerance 1e-2 * RMS, as for every bf16-input
forward.  A bf16 y carries its own rounding on top, up to half an ulp (2^-9
of |y|) per element, which alone exceeds 1e-2 * RMS wherever |y| > 5 RMS:
for bf16 output each element may also differ by 2^-8 |y_ref| (the rounding
bound with a factor 2 for the fp32 value it rounds).
"""
import numpy as np
import pytest

import oracle
from state_space_sequence_05_b300 import inputs as I

from _helpers import TOL, assert_close, to_device


def assert_close_bf16_out(got, ref, what=""):
    """max|got - ref| <= 1e-2 RMS(ref) + 2^-8 |ref|, elementwise."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    excess = np.abs(got - ref) - (TOL["bf16"] * rms + 2.0 ** -8 * np.abs(ref))
    worst = float(excess.max()) if excess.size else 0.0
    assert worst <= 0, f"{what}: exceeds the bf16-output bound by {worst:.3e} (RMS {rms:.3e})"

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _extras(fi, seed):
    """dt before its softplus (a raw projection value, bf16) and its per-head
    bias, and the gate z (bf16), all seeded."""
    rng = np.random.Generator(np.random.PCG64(seed))
    b, T, H, P = fi.x.shape
    dt_raw = I.bf16_round(rng.standard_normal((b, T, H), dtype=np.float32) * np.float32(0.5)
                          - np.float32(2.0))
    bias = rng.uniform(-2.0, 1.0, H).astype(np.float32)
    z = I.bf16_round(rng.standard_normal((b, T, H, P), dtype=np.float32) * np.float32(1.5))
    return dt_raw, bias, z


def _run(fi, softplus, gate, ybf16, seed=5):
    import torch
    from state_space_sequence_05_b300 import ssd
    d = to_device(fi)
    (dt_bits, dt_raw), bias, (z_bits, z) = _extras(fi, seed)
    dev = "cuda"
    dt_t = I.as_torch(dt_raw, dt_bits, dev, "bf16") if softplus else d["dt"]
    z_t = I.as_torch(z, z_bits, dev, "bf16") if gate else None
    bias_t = torch.from_numpy(bias).to(dev) if softplus else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    y, fin = ssd.ssd_chunk_scan_fwd(d["x"], dt_t, d["A"], d["B"], d["C"], d["D"], fi.wl.chunk,
                                    d["init"], d["cu"], dev_status=status, dt_bias=bias_t,
                                    dt_softplus=softplus, z=z_t,
                                    y_dtype=torch.bfloat16 if ybf16 else torch.float32)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert y.dtype == (torch.bfloat16 if ybf16 else torch.float32)
    dt_ref = oracle.softplus(dt_raw.astype(np.float64) + bias[None, None, :]) if softplus else fi.dt
    y_ref, fin_ref = oracle.ssd_scan(fi.x, dt_ref, fi.A, fi.B, fi.C, fi.D, fi.init,
                                     cu_seqlens=fi.cu_seqlens)
    if gate:
        y_ref = oracle.silu_gate(y_ref, z)
    return y.float().cpu().numpy(), fin.cpu().numpy(), y_ref, fin_ref


@pytest.mark.parametrize("softplus,gate,ybf16", [(True, False, False), (False, True, False),
                                                 (False, False, True), (True, True, True)])
def test_epilogue_options(softplus, gate, ybf16):
    """Each option alone and all three, two rows, several chunks and a ragged
    tail, two groups, nonzero init."""
    wl = I.small_workload(batch=2, seqlen=700, nheads=4, ngroups=2, chunk=256, seed=31)
    y, fin, y_ref, fin_ref = _run(I.make_forward_inputs(wl), softplus, gate, ybf16)
    if ybf16:
        assert_close_bf16_out(y, y_ref, "y")
    else:
        assert_close(y, y_ref, TOL["bf16"], "y")
    assert_close(fin, fin_ref, TOL["bf16"], "final")


def test_epilogue_varlen():
    wl = I.small_workload(batch=1, seqlen=0, nheads=4, ngroups=1, chunk=256, nseq=5, seed=32)
    fi = I.make_forward_inputs(wl)
    y, fin, y_ref, fin_ref = _run(fi, True, True, True)
    assert_close_bf16_out(y, y_ref, "y")
    assert_close(fin, fin_ref, TOL["bf16"], "final")


def test_epilogue_full_size_sampled_heads():
    """The benchmarked layer (b1 T8192 H80) with all three options; the oracle
    recomputes 6 heads."""
    fi = I.make_forward_inputs(I.WORKLOADS["l8k"])
    import torch
    from state_space_sequence_05_b300 import ssd
    d = to_device(fi)
    (dt_bits, dt_raw), bias, (z_bits, z) = _extras(fi, 9)
    dev = "cuda"
    y, fin = ssd.ssd_chunk_scan_fwd(d["x"], I.as_torch(dt_raw, dt_bits, dev, "bf16"), d["A"], d["B"],
                                    d["C"], d["D"], 256, d["init"], dt_bias=torch.from_numpy(bias).to(dev),
                                    dt_softplus=True, z=I.as_torch(z, z_bits, dev, "bf16"),
                                    y_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    y = y.float().cpu().numpy()
    fin = fin.cpu().numpy()
    for h in (0, 17, 33, 50, 66, 79):
        dt_h = oracle.softplus(dt_raw[:, :, h:h + 1].astype(np.float64) + bias[h])
        yr, fr = oracle.ssd_scan(fi.x[:, :, h:h + 1], dt_h, fi.A[h:h + 1], fi.B, fi.C, fi.D[h:h + 1],
                                 fi.init[:, h:h + 1])
        yr = oracle.silu_gate(yr, z[:, :, h:h + 1])
        assert_close_bf16_out(y[:, :, h:h + 1], yr, f"y head {h}")
        assert_close(fin[:, h:h + 1], fr, TOL["bf16"], f"final head {h}")


def test_epilogue_needs_the_tensor_core_shapes():
    """fp32 inputs run on the CUDA-core kernels, which have no fused epilogue:
    rejected on the host, nothing launched."""
    import torch
    from state_space_sequence_05_b300 import ssd
    wl = I.small_workload(batch=1, seqlen=64, nheads=2, headdim=16, dstate=16, ngroups=1,
                          chunk=64, dtype="f32", seed=3)
    d = to_device(I.make_forward_inputs(wl))
    before = ssd.kernel_launches()
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_chunk_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 64, d["init"],
                               dt_softplus=True)
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED
    assert ssd.kernel_launches() == before
