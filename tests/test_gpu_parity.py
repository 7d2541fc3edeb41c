"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs.  Tolerance: max|diff| <= tol * RMS(oracle) with
tol = 1e-4 for float32 inputs and 1e-2 for bfloat16 inputs, applied to y and
to the final states separately."""
import numpy as np
import pytest

import oracle
from state_space_sequence_05_b300 import inputs as I

from _helpers import (TOL, assert_close, gpu_seq, oracle_full, oracle_heads, oracle_workload,
                      run_gpu, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _check_full(fi, chunk=None, use_D=True):
    y, fin = run_gpu(fi, chunk=chunk, use_D=use_D)
    y_ref, fin_ref = oracle_full(fi, use_D=use_D)
    tol = TOL[fi.wl.dtype]
    ey = assert_close(y.cpu().numpy(), y_ref, tol, "y")
    ef = assert_close(fin.cpu().numpy(), fin_ref, tol, "final")
    return ey, ef


def test_tiny_fp32_workload():
    """b1 T256 H2 P16 N16 G1 chunk 64, float32 inputs, zero init."""
    _check_full(I.make_forward_inputs(I.WORKLOADS["tiny_fp32"]))


@pytest.mark.parametrize("chunk", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_bf16_small_ragged(chunk, G):
    """Several chunks plus a ragged tail (T = 300), two batch rows, groups
    1 / 2 / H, nonzero init."""
    wl = I.small_workload(batch=2, seqlen=300, nheads=4, ngroups=G, chunk=chunk, seed=100 + G)
    _check_full(I.make_forward_inputs(wl))


@pytest.mark.parametrize("P,N", [(1, 16), (16, 32), (64, 64), (128, 128), (32, 256)])
def test_fp32_shapes(P, N):
    wl = I.small_workload(batch=1, seqlen=200, nheads=2, headdim=P, dstate=N, ngroups=1,
                          chunk=64, dtype="f32", seed=200 + P)
    _check_full(I.make_forward_inputs(wl))


@pytest.mark.parametrize("T", [1, 37, 128, 129, 513])
def test_short_and_boundary_lengths(T):
    wl = I.small_workload(batch=2, seqlen=T, nheads=2, ngroups=1, chunk=128, seed=300 + T)
    _check_full(I.make_forward_inputs(wl))


def test_no_skip_term_and_zero_init():
    wl = I.small_workload(batch=1, seqlen=260, nheads=2, ngroups=1, init="zero", seed=9)
    _check_full(I.make_forward_inputs(wl), use_D=False)


def test_empty_sequence_batch_mode():
    import torch
    from state_space_sequence_05_b300 import ssd
    wl = I.small_workload(batch=2, seqlen=0, nheads=2, ngroups=1, seed=10)
    fi = I.make_forward_inputs(wl)
    d = to_device(fi)
    y, fin = ssd.ssd_chunk_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 128,
                                    d["init"])
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert np.array_equal(fin.cpu().numpy(), fi.init)


def _varlen_inputs(lens, H=4, P=64, N=128, G=2, dtype="bf16", seed=0, init=True):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    wl = I.Workload("varlen_test", 1, T, H, P, N, G, 128, dtype, "normal" if init else "zero")
    fi = I.make_forward_inputs(wl, seed=seed)
    fi.cu_seqlens = cu
    if init:
        fi.init = (rng.standard_normal((len(lens), H, P, N)) * 0.1).astype(np.float32)
    else:
        fi.init = None
    return fi


@pytest.mark.parametrize("init", [True, False])
@pytest.mark.parametrize("chunk", [64, 256])
def test_varlen_small(init, chunk):
    lens = [5, 0, 17, 1, 300, 129, 128, 256, 2]
    fi = _varlen_inputs(lens, seed=42, init=init)
    fi.wl = I.Workload(**{**fi.wl.__dict__, "chunk": chunk})
    _check_full(fi)


def test_varlen_malformed_cu_seqlens_reports_status():
    import torch
    from state_space_sequence_05_b300 import ssd
    fi = _varlen_inputs([10, 20, 30], seed=3)
    d = to_device(fi)
    bad = torch.tensor([0, 25, 20, 60], dtype=torch.int32, device="cuda")  # not monotone
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssd.ssd_chunk_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 128, d["init"], bad,
                           dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == ssd.SSD_ERR_INVALID
    # the same call with a valid array leaves the status at 0
    ssd.ssd_chunk_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 128, d["init"],
                           d["cu"], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_tensor_path_ignores_chunk_size_argument():
    """The tensor-core path always works in 128-token blocks (the tcgen05 tile
    height), whatever chunk_size asks: chunk 64 and 256 must give the oracle's
    result, and -- since the same blocks run -- the same bits."""
    wl = I.small_workload(batch=1, seqlen=1000, nheads=4, ngroups=1, seed=12)
    fi = I.make_forward_inputs(wl)
    y64, f64 = run_gpu(fi, chunk=64)
    y256, f256 = run_gpu(fi, chunk=256)
    y_ref, f_ref = oracle_full(fi)
    for y, f in ((y64, f64), (y256, f256)):
        assert_close(y.cpu().numpy(), y_ref, 1e-2, "y")
        assert_close(f.cpu().numpy(), f_ref, 1e-2, "final")
    assert np.array_equal(y64.cpu().numpy(), y256.cpu().numpy())


def test_chunk_size_independence_on_cuda_core_path():
    """The CUDA-core path honours chunk_size: fp32 inputs of the 2.7B head
    shape (P 64, N 128) at chunk 64, 128 and 256 each match the oracle at the
    fp32 bar and each other -- the block decomposition is an exact
    reordering of the recurrence ("Transformers are SSMs Review", sec. 3-2
    (4)), so only rounding may differ."""
    wl = I.small_workload(batch=2, seqlen=700, nheads=4, headdim=64, dstate=128, ngroups=2,
                          dtype="f32", seed=15)
    fi = I.make_forward_inputs(wl)
    y_ref, f_ref = oracle_full(fi)
    outs = {}
    for q in (64, 128, 256):
        y, f = run_gpu(fi, chunk=q)
        outs[q] = (y.cpu().numpy(), f.cpu().numpy())
        assert_close(outs[q][0], y_ref, TOL["f32"], f"y chunk {q}")
        assert_close(outs[q][1], f_ref, TOL["f32"], f"final chunk {q}")
    for q in (128, 256):
        assert_close(outs[q][0], outs[64][0], TOL["f32"], f"y chunk {q} vs 64")
        assert_close(outs[q][1], outs[64][1], TOL["f32"], f"final chunk {q} vs 64")
    assert not np.array_equal(outs[64][0], outs[256][0]), "chunk_size had no effect"


def test_split_carry_on_gpu():
    """One run over [0, T) equals [0, k) then [k, T) started from the first
    run's final state."""
    import torch
    from state_space_sequence_05_b300 import ssd
    wl = I.small_workload(batch=1, seqlen=700, nheads=4, ngroups=2, seed=13)
    fi = I.make_forward_inputs(wl)
    d = to_device(fi)
    k = 333
    y, fin = ssd.ssd_chunk_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 128,
                                    d["init"])
    sl = lambda t, a, b: t[:, a:b].contiguous()
    y1, f1 = ssd.ssd_chunk_scan_fwd(sl(d["x"], 0, k), sl(d["dt"], 0, k), d["A"], sl(d["B"], 0, k),
                                    sl(d["C"], 0, k), d["D"], 128, d["init"])
    y2, f2 = ssd.ssd_chunk_scan_fwd(sl(d["x"], k, 700), sl(d["dt"], k, 700), d["A"],
                                    sl(d["B"], k, 700), sl(d["C"], k, 700), d["D"], 128, f1)
    torch.cuda.synchronize()
    assert_close(torch.cat([y1, y2], 1).cpu().numpy(), y.cpu().numpy(), 1e-2, "split y")
    assert_close(f2.cpu().numpy(), fin.cpu().numpy(), 1e-2, "split final")


# ---- full-size workloads: every head (and every packed sequence) ----------

def _check_all(name):
    """The whole workload against the whole-problem oracle (fp64, all host
    threads): every batch row or packed sequence, every head."""
    fi = I.make_forward_inputs(I.WORKLOADS[name])
    y, fin = run_gpu(fi)
    y_ref, fin_ref = oracle_workload(name)
    tol = TOL[fi.wl.dtype]
    assert_close(y.cpu().numpy(), y_ref, tol, "y")
    assert_close(fin.cpu().numpy(), fin_ref, tol, "final")


def test_l2k_b4_all_heads():
    """b4 T2048 H80 P64 N128 G1 chunk 256, zero init."""
    _check_all("l2k_b4")


def test_l8k_all_heads():
    """b1 T8192 H80 P64 N128 G1 chunk 256, init ~ N(0, 0.1^2)."""
    _check_all("l8k")


def test_l64k_all_heads():
    """b1 T65536, same layer."""
    _check_all("l64k")


def test_varlen64_all_sequences_and_heads():
    """64 packed sequences, lengths log-uniform in [64, 8192], H64 G8."""
    _check_all("varlen64")


# ---- decode ----------------------------------------------------------------

def _decode_run(wl, rows, steps):
    import torch
    from state_space_sequence_05_b300 import ssd
    dec = I.make_decode_inputs(wl)
    dev = torch.device("cuda")
    state = torch.from_numpy(dec.state0).to(dev)
    A = torch.from_numpy(dec.A).to(dev)
    D = torch.from_numpy(dec.D).to(dev)
    ref_state = dec.state0[rows].astype(np.float64)
    ys, refs = [], []
    for t in range(steps):
        tok = I.make_decode_token(wl, dec, t)
        y = ssd.ssd_state_update(state, I.as_torch(tok.x, tok.bits["x"], dev, "bf16"),
                                 I.as_torch(tok.dt, tok.bits["dt"], dev, "bf16"), A,
                                 I.as_torch(tok.B, tok.bits["B"], dev, "bf16"),
                                 I.as_torch(tok.C, tok.bits["C"], dev, "bf16"), D)
        yr, ref_state = oracle.ssd_step(ref_state, tok.x[rows], tok.dt[rows], dec.A, tok.B[rows],
                                        tok.C[rows], dec.D)
        ys.append(y[rows].cpu().numpy())
        refs.append(yr)
    torch.cuda.synchronize()
    return np.stack(ys), np.stack(refs), state[rows].cpu().numpy(), ref_state


def test_decode_b256_128_steps_every_8th_row():
    """b256 H80 P64 N128, fp32 state updated in place over 128 steps; every
    8th batch row and the last one followed by the oracle step by step (all
    heads of each; the oracle step is single-threaded)."""
    wl = I.DECODE_WORKLOADS["decode_b256"]
    rows = list(range(0, wl.batch, 8)) + [wl.batch - 1]
    ys, refs, st, st_ref = _decode_run(wl, rows, wl.steps)
    assert_close(ys, refs, 1e-2, "decode y")
    assert_close(st, st_ref, 1e-2, "decode state")


@pytest.mark.parametrize("N,G", [(16, 1), (64, 2), (256, 4)])
def test_decode_shapes_all_rows(N, G):
    wl = I.DecodeWorkload("dec_small", 3, 4, 24, N, G, 5)
    ys, refs, st, st_ref = _decode_run(wl, [0, 1, 2], wl.steps)
    assert_close(ys, refs, 1e-2, "decode y")
    assert_close(st, st_ref, 1e-2, "decode state")


def test_decode_steps_equal_forward():
    """128 single-token steps from init equal one forward over the same 128
    tokens with the same init."""
    import torch
    from state_space_sequence_05_b300 import ssd
    wl = I.small_workload(batch=2, seqlen=128, nheads=4, ngroups=2, seed=14)
    fi = I.make_forward_inputs(wl)
    d = to_device(fi)
    y, fin = ssd.ssd_chunk_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 128,
                                    d["init"])
    state = d["init"].clone()
    ys = []
    for t in range(128):
        ys.append(ssd.ssd_state_update(state, d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(),
                                       d["A"], d["B"][:, t].contiguous(),
                                       d["C"][:, t].contiguous(), d["D"]))
    torch.cuda.synchronize()
    assert_close(torch.stack(ys, 1).cpu().numpy(), y.cpu().numpy(), 1e-2, "decode vs fwd y")
    assert_close(state.cpu().numpy(), fin.cpu().numpy(), 1e-2, "decode vs fwd state")


def _with_decay(fi, A, dt_per_head, rng):
    """The same inputs with A and dt replaced: dt[h] ~ dt_per_head[h] x (1 +/- 10%),
    rounded to bf16 like every bf16 input."""
    A = np.asarray(A, np.float32)
    b, T, H = fi.dt.shape
    dt = (np.asarray(dt_per_head, np.float32)[None, None, :] *
          (1.0 + 0.1 * rng.uniform(-1, 1, (b, T, H)))).astype(np.float32)
    fi.A = A
    fi.bits["dt"], fi.dt = I.bf16_round(dt)
    return fi


def test_decay_regimes_on_the_tensor_path():
    """One head per decay regime of the tensor-core mask: a chunk whose whole
    decay fits the exp(-cum) dt table (dt 0.03), chunks too strong for the
    table but with 32-token blocks that still factor (dt 0.08), blocks whose
    own decay needs one exponential per entry (dt 0.3), and a nearly
    undamped head (dt 1e-3).  A = -16 on every head."""
    wl = I.small_workload(batch=2, seqlen=700, nheads=4, ngroups=2, chunk=128, seed=21)
    fi = _with_decay(I.make_forward_inputs(wl), [-16.0] * 4, [0.03, 0.08, 0.3, 1e-3],
                     np.random.default_rng(21))
    _check_full(fi)


def test_zero_decay_is_linear_attention_on_gpu():
    """A = 0: no decay at all (the mask is the causal C B^T dt)."""
    wl = I.small_workload(batch=1, seqlen=600, nheads=4, ngroups=1, chunk=128, seed=22)
    fi = _with_decay(I.make_forward_inputs(wl), [0.0] * 4, [0.01, 0.02, 0.05, 0.1],
                     np.random.default_rng(22))
    _check_full(fi)


@pytest.mark.parametrize("batch,T", [(3, 1500), (1, 4096), (6, 640)])
def test_segment_lengths_chosen_per_shape(batch, T):
    """Dense batches pick their segment length from the SM count and the
    shape; each pick must give the same function."""
    wl = I.small_workload(batch=batch, seqlen=T, nheads=8, ngroups=2, chunk=256,
                          seed=400 + T)
    fi = I.make_forward_inputs(wl)
    heads = [0, 5]
    y, fin = run_gpu(fi)
    ref = oracle_heads(fi, heads)
    y_np, f_np = y.cpu().numpy(), fin.cpu().numpy()
    for (s, h), (yr, fr) in ref.items():
        assert_close(gpu_seq(fi, y_np, s, h), yr, TOL["bf16"], f"y s{s} h{h}")
        assert_close(f_np[s, h], fr, TOL["bf16"], f"final s{s} h{h}")
