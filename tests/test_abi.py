"""The C-ABI library loads, exports every symbol include/ssd.h declares, and
rejects bad arguments on the host before touching the GPU (CPU only: no
compute call here needs a device)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from state_space_sequence_05_b300 import ssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build_library()
    return ssd.load_library()


def _declared():
    text = open(os.path.join(ROOT, "include", "ssd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = _declared()
    assert {"ssd_chunk_scan_fwd", "ssd_state_update", "ssd_chunk_scan_fwd_workspace_size",
            "ssd_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ssd.h but not exported"
    assert set(names) == set(ssd.SIGNATURES), "binding signatures out of sync with the header"


def test_status_strings(lib):
    assert ssd.status_string(0) == "ok"
    assert "timed out" in ssd.status_string(4)
    assert ssd.version() >= 100


def test_workspace_query(lib):
    n = ssd.ssd_chunk_scan_fwd_workspace_size(1, 8192, 80, 64, 128, 1, 256, ssd.SSD_DT_BF16)
    assert 0 < n < (1 << 30)
    assert ssd.ssd_chunk_scan_fwd_workspace_size(1, 0, 2, 16, 16, 1, 64, ssd.SSD_DT_F32,
                                                 True, 0) == 0
    with pytest.raises(ssd.SSDError):
        ssd.ssd_chunk_scan_fwd_workspace_size(1, 100, 3, 16, 16, 2, 64, ssd.SSD_DT_F32)  # H%G
    with pytest.raises(ssd.SSDError):
        ssd.ssd_chunk_scan_fwd_workspace_size(1, 100, 2, 16, 16, 1, 96, ssd.SSD_DT_F32)  # chunk
    with pytest.raises(ssd.SSDError):
        ssd.ssd_chunk_scan_fwd_workspace_size(1, 100, 2, 16, 24, 1, 64, ssd.SSD_DT_F32)  # dstate


def _fwd(lib, **kw):
    a = dict(x=None, dt=None, A=None, B=None, C=None, D=None, batch=1, seqlen=16, nheads=2,
             headdim=16, dstate=16, ngroups=1, chunk=64, dtype=0, init=None, cu=None, nseq=0,
             y=None, final=None, ws=None, ws_bytes=0, status=None, stream=None)
    a.update(kw)
    return lib.ssd_chunk_scan_fwd(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["batch"],
                                  a["seqlen"], a["nheads"], a["headdim"], a["dstate"],
                                  a["ngroups"], a["chunk"], a["dtype"], a["init"], a["cu"],
                                  a["nseq"], a["y"], a["final"], a["ws"], a["ws_bytes"],
                                  a["status"], a["stream"])


def test_host_side_rejections(lib):
    fake = ctypes.c_void_p(0x10000)        # never dereferenced: checks fail first
    odd = ctypes.c_void_p(0x10008)         # not 16-byte aligned
    ptrs = dict(x=fake, dt=fake, A=fake, B=fake, C=fake, y=fake)
    assert _fwd(lib) == ssd.SSD_ERR_INVALID                             # null pointers
    assert _fwd(lib, **ptrs, dtype=7) == ssd.SSD_ERR_INVALID            # bad dtype
    assert _fwd(lib, **ptrs, nheads=3, ngroups=2) == ssd.SSD_ERR_INVALID
    assert _fwd(lib, **ptrs, chunk=32) == ssd.SSD_ERR_UNSUPPORTED
    assert _fwd(lib, **ptrs, headdim=129) == ssd.SSD_ERR_UNSUPPORTED
    assert _fwd(lib, **ptrs, dstate=48) == ssd.SSD_ERR_UNSUPPORTED
    assert _fwd(lib, **{**ptrs, "x": odd}) == ssd.SSD_ERR_INVALID        # misaligned
    assert _fwd(lib, **ptrs, batch=2, cu=fake, nseq=1) == ssd.SSD_ERR_INVALID
    assert _fwd(lib, **ptrs, seqlen=-1) == ssd.SSD_ERR_INVALID
    # workspace present but too small
    assert _fwd(lib, **ptrs, ws=fake, ws_bytes=16) == ssd.SSD_ERR_INVALID
    assert lib.ssd_state_update(None, fake, fake, fake, fake, fake, None, 1, 2, 16, 16, 1, 0,
                                fake, None) == ssd.SSD_ERR_INVALID
    assert lib.ssd_state_update(fake, fake, fake, fake, fake, fake, None, 1, 2, 16, 20, 1, 0,
                                fake, None) == ssd.SSD_ERR_UNSUPPORTED
    assert lib.ssd_state_update(fake, fake, fake, fake, fake, fake, None, 1, 3, 16, 16, 2, 0,
                                fake, None) == ssd.SSD_ERR_INVALID


def test_binding_fails_loudly_without_library(tmp_path):
    saved = ssd._lib
    ssd._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            ssd.load_library(str(tmp_path / "nope.so"))
    finally:
        ssd._lib = saved


def test_host_side_rejections_of_the_other_entry_points(lib):
    """The fused-epilogue forward, the backward, the context-parallel steps and
    the selective scan check their arguments on the host before any CUDA call
    (so this runs without a GPU)."""
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    E = ssd.FwdEpilogue

    def fwd_ex(epi, dtype=0, P=16, N=16, z=None):
        e = E(None, epi.get("softplus", 0), z, epi.get("bf16", 0))
        return lib.ssd_chunk_scan_fwd_ex(fake, fake, fake, fake, fake, None, 1, 16, 2, P, N, 1, 64,
                                         dtype, None, None, 0, fake, None, None, 0, None, None,
                                         ctypes.byref(e))
    # the fused epilogue exists on the tensor-core shapes only
    assert fwd_ex({"softplus": 1}) == ssd.SSD_ERR_UNSUPPORTED
    assert fwd_ex({"bf16": 1}, dtype=0, P=64, N=128) == ssd.SSD_ERR_UNSUPPORTED
    # z must be 16-byte aligned
    assert fwd_ex({}, dtype=1, P=64, N=128, z=odd) == ssd.SSD_ERR_INVALID

    def bwd(dtype=0, H=2, P=16, N=16, G=1, ws=None, ws_bytes=0):
        return lib.ssd_chunk_scan_bwd(fake, fake, fake, fake, fake, None, 1, 16, H, P, N, G, dtype,
                                      None, fake, None, fake, fake, fake, fake, fake, None, None,
                                      ws, ws_bytes, None, None)
    assert bwd(dtype=7) == ssd.SSD_ERR_INVALID
    assert bwd(H=3, G=2) == ssd.SSD_ERR_INVALID
    assert bwd(P=129, N=128) == ssd.SSD_ERR_UNSUPPORTED
    assert bwd() == ssd.SSD_ERR_INVALID                                   # no workspace
    need = lib.ssd_chunk_scan_bwd_workspace_size(1, 16, 2, 16, 16, 1, 0)
    assert 0 < need < (1 << 30)
    assert bwd(ws=fake, ws_bytes=need - 1) == ssd.SSD_ERR_INVALID         # too small
    assert lib.ssd_chunk_scan_bwd_workspace_size(1, 16, 2, 129, 128, 1, 0) == ctypes.c_size_t(-1).value

    assert lib.ssd_segment_decay(fake, fake, 1, 16, 0, 0, fake, None) == ssd.SSD_ERR_INVALID
    assert lib.ssd_segment_decay(None, fake, 1, 16, 2, 0, fake, None) == ssd.SSD_ERR_INVALID
    assert lib.ssd_segment_combine(fake, None, None, 2, 1, 2, 4, 4, fake, None) == ssd.SSD_ERR_INVALID
    assert lib.ssd_segment_combine(fake, fake, None, 2, 1, 2, 0, 4, fake, None) == ssd.SSD_ERR_INVALID

    def s6(batch=1, N=16, x=fake):
        return lib.ssd_selective_scan_fwd(x, fake, fake, fake, fake, None, None, batch, 16, 8, N,
                                          0, fake, None, None)
    assert s6(N=24) == ssd.SSD_ERR_UNSUPPORTED
    assert s6(batch=70000) == ssd.SSD_ERR_UNSUPPORTED
    assert s6(x=None) == ssd.SSD_ERR_INVALID
