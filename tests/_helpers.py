"""Shared helpers for the parity tests: move seeded inputs to the GPU, run the
library through its binding, run the oracle (whole problem or sampled
heads), and compare with the tolerance metric max|diff| <= tol * RMS(ref).

Tolerances: 1e-4 for float32 inputs, 1e-2 for bfloat16 inputs (fp32 state
and accumulation).  The pages give none; these are the targets the library
is held to, applied to y and, separately, to the final states.
"""
from __future__ import annotations

import functools

import numpy as np

import oracle
from state_space_sequence_05_b300 import inputs as I

TOL = {"f32": 1e-4, "bf16": 1e-2}


def to_device(fi: I.ForwardInputs, device="cuda"):
    import torch
    dtype = fi.wl.dtype
    d = {
        "x": I.as_torch(fi.x, fi.bits.get("x"), device, dtype),
        "dt": I.as_torch(fi.dt, fi.bits.get("dt"), device, dtype),
        "B": I.as_torch(fi.B, fi.bits.get("B"), device, dtype),
        "C": I.as_torch(fi.C, fi.bits.get("C"), device, dtype),
        "A": torch.from_numpy(fi.A).to(device),
        "D": torch.from_numpy(fi.D).to(device),
        "init": None if fi.init is None else torch.from_numpy(fi.init).to(device),
        "cu": None if fi.cu_seqlens is None else torch.from_numpy(fi.cu_seqlens).to(device),
    }
    return d


def run_gpu(fi: I.ForwardInputs, chunk=None, use_D=True, device="cuda"):
    """Run the forward through the binding; the device status must stay 0
    (a bounded wait that expired would report SSD_ERR_TIMEOUT there)."""
    import torch
    from state_space_sequence_05_b300 import ssd
    d = to_device(fi, device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    y, fin = ssd.ssd_chunk_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"],
                                    d["D"] if use_D else None, chunk or fi.wl.chunk, d["init"],
                                    d["cu"], dev_status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, f"device status {st} ({ssd.status_string(st)})"
    return y, fin


def oracle_full(fi: I.ForwardInputs, use_D=True):
    return oracle.ssd_scan(fi.x, fi.dt, fi.A, fi.B, fi.C, fi.D if use_D else None, fi.init,
                           cu_seqlens=fi.cu_seqlens)


@functools.lru_cache(maxsize=4)
def oracle_workload(name: str):
    """The whole-problem oracle of a named workload, computed once per test
    session (several kernels are checked against it)."""
    fi = I.make_forward_inputs(I.WORKLOADS[name])
    return oracle_full(fi)


def oracle_heads(fi: I.ForwardInputs, heads, seqs=None):
    """Oracle for a subset of heads (and, for varlen, of sequences): returns
    {(s, h): (y_seq [len, P], final [P, N])}."""
    H, G = fi.wl.nheads, fi.wl.ngroups
    out = {}
    nseq = fi.nseq
    seqs = range(nseq) if seqs is None else seqs
    for h in heads:
        g = h * G // H
        for s in seqs:
            if fi.cu_seqlens is None:
                bsl = slice(s, s + 1)
                tsl = slice(None)
            else:
                bsl = slice(0, 1)
                tsl = slice(int(fi.cu_seqlens[s]), int(fi.cu_seqlens[s + 1]))
            init = None if fi.init is None else fi.init[s:s + 1, h:h + 1]
            y, fin = oracle.ssd_scan(fi.x[bsl, tsl, h:h + 1], fi.dt[bsl, tsl, h:h + 1],
                                     fi.A[h:h + 1], fi.B[bsl, tsl, g:g + 1], fi.C[bsl, tsl, g:g + 1],
                                     fi.D[h:h + 1], init)
            out[(s, h)] = (y[0, :, 0, :], fin[0, 0])
    return out


def gpu_seq(fi: I.ForwardInputs, y_np, s, h):
    if fi.cu_seqlens is None:
        return y_np[s, :, h, :]
    return y_np[0, int(fi.cu_seqlens[s]):int(fi.cu_seqlens[s + 1]), h, :]


def assert_close(got, ref, tol, what=""):
    e = oracle.rel_err(got, ref)
    assert e <= tol, f"{what}: max|diff|/RMS = {e:.3e} > {tol:.1e}"
    return e
