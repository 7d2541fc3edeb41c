"""The bounded device waits of the tensor-core forward and backward run out
cleanly.

Every wait in the kernels (an mbarrier phase, a predecessor's hand-off flag)
gives up after a time limit, records SSD_ERR_TIMEOUT in dev_status and lets
the kernel unwind with its tensor memory freed -- no trap, no fault.  Here a
test hook shortens the limit to 2 ms and holds back one signal of work unit
0: in the fused and pipelined kernels its hand-off flag (the segment end
state it should publish), so the unit waiting for it runs out; in the split
kernels its first decay mask, so the MMA issuer waiting for it runs out.
The call must return, report the timeout, and leave the context usable: the
next call on the same stream, with the hook off, is exact.
"""
import os

import pytest

from state_space_sequence_05_b300 import inputs as I

from _helpers import TOL, assert_close, oracle_full, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(params=["fused", "pipelined", "split"])
def kernel(request, monkeypatch):
    """Every tensor-core forward takes the hook."""
    monkeypatch.setenv("SSD_TC_KERNEL", request.param)
    return request.param


def test_held_hand_off_times_out_then_next_call_is_exact(kernel):
    import torch
    from state_space_sequence_05_b300 import ssd
    # 16 chunks of 128 tokens per head: several segments, so unit 0 (first
    # segment of head 0) has a successor that waits for its end state
    wl = I.small_workload(batch=1, seqlen=2048, nheads=4, ngroups=1, chunk=256, seed=31)
    fi = I.make_forward_inputs(wl)
    d = to_device(fi)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 256, d["init"])
    try:
        ssd.test_set_forward_wait(2_000_000, 0)
        ssd.ssd_chunk_scan_fwd(*args, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == ssd.SSD_ERR_TIMEOUT
    finally:
        ssd.test_set_forward_wait(0, -1)
    y, fin = ssd.ssd_chunk_scan_fwd(*args, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y_ref, f_ref = oracle_full(fi)
    assert_close(y.cpu().numpy(), y_ref, TOL["bf16"], "y after the expired call")
    assert_close(fin.cpu().numpy(), f_ref, TOL["bf16"], "final after the expired call")


@pytest.mark.parametrize("hold", [1, 2], ids=["gradients", "state_scan"])
def test_backward_held_mma_completion_times_out_then_next_call_is_exact(hold):
    """The tensor-core backward: one MMA completion of the gradient kernel
    (hold 1) or of the state scans (hold 2) is never signalled, so the
    threads waiting for it give up after the hook's poll bound and the call
    reports SSD_ERR_TIMEOUT; the next call, hook off, matches the fp64
    backward oracle."""
    import numpy as np
    import torch
    import oracle
    from state_space_sequence_05_b300 import ssd
    wl = I.small_workload(batch=1, seqlen=192, nheads=2, headdim=64, dstate=128, ngroups=1,
                          chunk=128, dtype="bf16", seed=33)
    fi = I.make_forward_inputs(wl)
    d = to_device(fi)
    rng = np.random.Generator(np.random.PCG64(933))
    dy = rng.standard_normal(fi.x.shape).astype(np.float32)
    dyt = torch.from_numpy(dy).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], dyt)
    try:
        ssd.test_set_backward_wait(20000, hold)
        ssd.ssd_chunk_scan_bwd(*args, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == ssd.SSD_ERR_TIMEOUT
    finally:
        ssd.test_set_backward_wait(0, 0)
    g = ssd.ssd_chunk_scan_bwd(*args, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.ssd_bwd(fi.x, fi.dt, fi.A, fi.B, fi.C, fi.D, fi.init, dy, None)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD", "dinit"):
        e = oracle.rel_err(g[k].cpu().numpy(), ref[k])
        assert e <= 1e-3, f"{k} after the expired call: max|diff|/RMS = {e:.3e}"
