"""The split tensor-core forward and the states-only pass against the fp64
oracle.

SSD_TC_KERNEL=split runs the bf16 / headdim 64 / dstate 128 forward as
separate kernels: the chunks' decay tables, the segment states (each
segment's end state from a zero state), the state passing over segments
and the outputs from each segment's entering state.  ssd_chunk_scan_states
runs all of that but the outputs.  Tolerances as in the other parity tests:
max|diff| <= tol * RMS(oracle), tol = 1e-2 for bfloat16 and 1e-4 for
float32 inputs.
"""
import numpy as np
import pytest

import oracle
from state_space_sequence_05_b300 import inputs as I

from _helpers import TOL, assert_close, oracle_full, oracle_workload, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture
def split(monkeypatch):
    monkeypatch.setenv("SSD_TC_KERNEL", "split")


def _check(fi):
    y, fin = run_gpu(fi)
    y_ref, fin_ref = oracle_full(fi)
    tol = TOL[fi.wl.dtype]
    assert_close(y.cpu().numpy(), y_ref, tol, "y")
    assert_close(fin.cpu().numpy(), fin_ref, tol, "final")


@pytest.mark.parametrize("batch,T,H,G,seed", [
    (1, 1, 1, 1, 1),        # one token
    (1, 128, 1, 1, 2),      # exactly one chunk
    (2, 129, 2, 1, 3),      # one chunk and one token
    (2, 300, 4, 2, 4),      # ragged tail
    (2, 1000, 4, 1, 5),     # several segments
    (3, 2048, 8, 2, 6),     # 16 chunks per row
])
def test_split_forward_small(split, batch, T, H, G, seed):
    wl = I.small_workload(batch=batch, seqlen=T, nheads=H, ngroups=G, chunk=128, seed=900 + seed)
    _check(I.make_forward_inputs(wl))


@pytest.mark.parametrize("init", ["zero", "normal"])
def test_split_forward_varlen(split, init):
    """Packed sequences with an empty one, one shorter than a chunk and
    lengths across segment boundaries."""
    lens = [5, 0, 130, 64, 1500, 257, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    wl = I.Workload("split_varlen", 1, int(cu[-1]), 4, 64, 128, 2, 128, "bf16", init, seed=911)
    fi = I.make_forward_inputs(wl)
    fi.cu_seqlens = cu
    if init == "normal":
        fi.init = (np.random.default_rng(912).standard_normal((len(lens), 4, 64, 128)) *
                   0.1).astype(np.float32)
    _check(fi)


@pytest.mark.parametrize("name", ["l2k_b4", "l8k", "varlen64"])
def test_split_forward_full_size(split, name):
    """Every head (every packed sequence) of the full-size workloads."""
    fi = I.make_forward_inputs(I.WORKLOADS[name])
    y, fin = run_gpu(fi)
    y_ref, fin_ref = oracle_workload(name)
    assert_close(y.cpu().numpy(), y_ref, TOL["bf16"], "y")
    assert_close(fin.cpu().numpy(), fin_ref, TOL["bf16"], "final")


def _states(fi, d):
    from state_space_sequence_05_b300 import ssd
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fin = ssd.ssd_chunk_scan_states(d["x"], d["dt"], d["A"], d["B"], fi.wl.chunk, d["init"],
                                    d["cu"], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return fin.cpu().numpy()


@pytest.mark.parametrize("case", ["bf16_batch", "bf16_varlen", "f32_generic"])
def test_states_only_pass(case):
    """The final states of ssd_chunk_scan_states against the oracle (the
    tensor-core shapes on the segment-state kernels, a float32 shape on the
    CUDA-core forward)."""
    if case == "bf16_batch":
        wl = I.small_workload(batch=2, seqlen=1500, nheads=4, ngroups=2, chunk=256, seed=921)
        fi = I.make_forward_inputs(wl)
    elif case == "bf16_varlen":
        lens = [700, 0, 3, 1100, 128]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        wl = I.Workload("states_varlen", 1, int(cu[-1]), 4, 64, 128, 1, 256, "bf16", "zero",
                        seed=922)
        fi = I.make_forward_inputs(wl)
        fi.cu_seqlens = cu
        fi.init = (np.random.default_rng(923).standard_normal((len(lens), 4, 64, 128)) *
                   0.1).astype(np.float32)
    else:
        wl = I.small_workload(batch=2, seqlen=333, nheads=3, headdim=16, dstate=32, ngroups=1,
                              chunk=64, dtype="f32", seed=924)
        fi = I.make_forward_inputs(wl)
    d = to_device(fi)
    fin = _states(fi, d)
    _, fin_ref = oracle_full(fi)
    assert_close(fin, fin_ref, TOL[fi.wl.dtype], "states-only final")


def test_states_only_pass_l8k():
    """The full-size layer: final state against the oracle."""
    fi = I.make_forward_inputs(I.WORKLOADS["l8k"])
    d = to_device(fi)
    fin = _states(fi, d)
    _, fin_ref = oracle_workload("l8k")
    assert_close(fin, fin_ref, TOL["bf16"], "states-only final")
