"""ssd_chunk_scan_fwd_noalloc: the forward for callers that cannot allocate
device memory (a plugin in a framework that owns all device memory, a loop
where an allocation is not allowed).  It keeps its scratch in a fixed array
inside the library instead of a caller-provided workspace.

Checked through the C ABI on calls in a row -- so that whatever the previous
call left in the shared scratch array is seen by the next one -- against the
fp64 oracle at the build's tolerances and against the workspace entry point.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import oracle
from state_space_sequence_05_b300 import inputs as I

from _helpers import TOL, assert_close, oracle_full, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()
    from state_space_sequence_05_b300 import ssd
    return ssd.load_library()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, fi, d, y, fin, status):
    import torch
    from state_space_sequence_05_b300 import ssd
    wl = fi.wl
    b, T, H, P = d["x"].shape
    G, N = d["B"].shape[2], d["B"].shape[3]
    code = ssd.SSD_DT_BF16 if wl.dtype == "bf16" else ssd.SSD_DT_F32
    return lib.ssd_chunk_scan_fwd_noalloc(
        _p(d["x"]), _p(d["dt"]), _p(d["A"]), _p(d["B"]), _p(d["C"]), _p(d["D"]), b, T, H, P, N,
        G, wl.chunk, code, _p(d["init"]), _p(d["cu"]), fi.nseq, _p(y), _p(fin), _p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _problem(name):
    if name == "f32":
        return I.make_forward_inputs(I.small_workload(batch=1, seqlen=300, nheads=2, headdim=16,
                                                      dstate=16, ngroups=1, chunk=64,
                                                      dtype="f32", seed=501))
    if name == "varlen":
        # several packed sequences, one of them empty and one shorter than a chunk
        lens = [5, 0, 130, 64, 257]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        wl = I.Workload("noalloc_varlen", 1, int(cu[-1]), 4, 32, 64, 2, 64, "f32", "normal",
                        seed=503)
        fi = I.make_forward_inputs(wl)
        fi.cu_seqlens = cu
        fi.init = (np.random.default_rng(503).standard_normal((len(lens), 4, 32, 64)) *
                   0.1).astype(np.float32)
        return fi
    return I.make_forward_inputs(I.small_workload(batch=2, seqlen=260, nheads=4, headdim=64,
                                                  dstate=128, ngroups=2, chunk=128,
                                                  dtype="bf16", seed=502))


def test_noalloc_matches_oracle_on_calls_in_a_row(lib):
    import torch
    from state_space_sequence_05_b300 import ssd
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for name in ("f32", "bf16", "varlen", "f32", "varlen"):
        fi = _problem(name)
        d = to_device(fi)
        y_ws, f_ws = ssd.ssd_chunk_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                            fi.wl.chunk, d["init"], d["cu"])
        y = torch.full_like(y_ws, float("nan"))
        fin = torch.full_like(f_ws, float("nan"))
        st = _noalloc(lib, fi, d, y, fin, status)
        assert st == ssd.SSD_OK, ssd.status_string(st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        tol = TOL[fi.wl.dtype]
        y_ref, f_ref = oracle_full(fi)
        assert_close(y.cpu().numpy(), y_ref, tol, f"{name} y vs oracle")
        assert_close(fin.cpu().numpy(), f_ref, tol, f"{name} final vs oracle")
        assert_close(y.cpu().numpy(), y_ws.cpu().numpy(), tol, f"{name} y vs workspace call")
        assert_close(fin.cpu().numpy(), f_ws.cpu().numpy(), tol, f"{name} final vs workspace call")


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    """An oversized problem is refused on the host: nothing is launched, and
    neither the outputs nor the status word are touched."""
    import torch
    from state_space_sequence_05_b300 import ssd
    # 128 chunks x 8 heads x 64 x 128 fp32 states = 32 MiB of scratch > 16 MiB
    dev = "cuda"
    x = torch.zeros((1, 8192, 8, 64), device=dev)
    dt = torch.zeros((1, 8192, 8), device=dev)
    A = torch.zeros(8, device=dev)
    Bm = torch.zeros((1, 8192, 1, 128), device=dev)
    y = torch.full_like(x, float("nan"))
    fin = torch.full((1, 8, 64, 128), float("nan"), device=dev)
    status = torch.full((1,), 12345, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    launches = ssd.kernel_launches()
    st = lib.ssd_chunk_scan_fwd_noalloc(_p(x), _p(dt), _p(A), _p(Bm), _p(Bm), None, 1, 8192, 8,
                                        64, 128, 1, 64, ssd.SSD_DT_F32, None, None, 0, _p(y),
                                        _p(fin), _p(status), None)
    torch.cuda.synchronize()
    assert st == ssd.SSD_ERR_UNSUPPORTED
    assert ssd.kernel_launches() == launches
    assert int(status.item()) == 12345
    assert torch.isnan(y).all() and torch.isnan(fin).all()
