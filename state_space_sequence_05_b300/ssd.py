"""Python binding of libssd_b300.so (ctypes): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this
module checks tensor placement and dtypes, allocates outputs and the
workspace with PyTorch, passes raw device pointers and the current CUDA
stream, and turns status codes into exceptions.  There is no fallback: if
the library is missing or fails to load, every call raises.

Function names follow the C entry points in include/ssd.h.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssd_b300.so")

SSD_OK, SSD_ERR_INVALID, SSD_ERR_UNSUPPORTED, SSD_ERR_CUDA, SSD_ERR_TIMEOUT = range(5)
SSD_DT_F32, SSD_DT_BF16 = 0, 1

# Names and C signatures of every symbol include/ssd.h declares.
_vp, _fp, _ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_ci, _sz = ctypes.c_int, ctypes.c_size_t


class FwdEpilogue(ctypes.Structure):
    """ssd_fwd_epilogue_t: the fused epilogue options of ssd_chunk_scan_fwd_ex."""
    _fields_ = [("dt_bias", ctypes.c_void_p), ("dt_softplus", ctypes.c_int),
                ("z", ctypes.c_void_p), ("y_bf16", ctypes.c_int)]

SIGNATURES = {
    "ssd_chunk_scan_fwd": (_ci, [_vp, _vp, _fp, _vp, _vp, _fp, _ci, _ci, _ci, _ci, _ci, _ci, _ci,
                                 _ci, _fp, _ip, _ci, _fp, _fp, _vp, _sz, _ip, _vp]),
    "ssd_chunk_scan_fwd_ex": (_ci, [_vp, _vp, _fp, _vp, _vp, _fp, _ci, _ci, _ci, _ci, _ci, _ci,
                                    _ci, _ci, _fp, _ip, _ci, _vp, _fp, _vp, _sz, _ip, _vp,
                                    ctypes.POINTER(FwdEpilogue)]),
    "ssd_chunk_scan_fwd_noalloc": (_ci, [_vp, _vp, _fp, _vp, _vp, _fp, _ci, _ci, _ci, _ci, _ci,
                                         _ci, _ci, _ci, _fp, _ip, _ci, _fp, _fp, _ip, _vp]),
    "ssd_chunk_scan_fwd_workspace_size": (_sz, [_ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci]),
    "ssd_chunk_scan_states_workspace_size": (_sz, [_ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci,
                                                   _ci]),
    "ssd_chunk_scan_states": (_ci, [_vp, _vp, _fp, _vp, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _ci, _fp,
                                    _ip, _ci, _fp, _vp, _sz, _ip, _vp]),
    "ssd_state_update": (_ci, [_fp, _vp, _vp, _fp, _vp, _vp, _fp, _ci, _ci, _ci, _ci, _ci, _ci,
                               _fp, _vp]),
    "ssd_selective_scan_fwd": (_ci, [_vp, _vp, _fp, _vp, _vp, _fp, _fp, _ci, _ci, _ci, _ci, _ci,
                                     _fp, _fp, _vp]),
    "ssd_chunk_scan_bwd_workspace_size": (_sz, [_ci, _ci, _ci, _ci, _ci, _ci, _ci]),
    "ssd_chunk_scan_bwd": (_ci, [_vp, _vp, _fp, _vp, _vp, _fp, _ci, _ci, _ci, _ci, _ci, _ci, _ci,
                                 _fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, _vp, _sz, _ip,
                                 _vp]),
    "ssd_segment_decay": (_ci, [_vp, _fp, _ci, _ci, _ci, _ci, _fp, _vp]),
    "ssd_segment_combine": (_ci, [_fp, _fp, _fp, _ci, _ci, _ci, _ci, _ci, _fp, _vp]),
    "ssd_status_string": (ctypes.c_char_p, [_ci]),
    "ssd_version": (_ci, []),
    "ssd_kernel_launches": (ctypes.c_uint64, []),
    "ssd_test_set_forward_wait": (None, [ctypes.c_ulonglong, _ci]),
    "ssd_test_set_backward_wait": (None, [ctypes.c_ulonglong, _ci]),
}

_lib = None


class SSDError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load_library(path: str = LIB_PATH):
    """Load the CUDA library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -m state_space_sequence_05_b300._build "
            "or __graft_entry__.build()); there is no non-CUDA implementation")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().ssd_status_string(int(status)).decode()


def version() -> int:
    return int(load_library().ssd_version())


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load_library().ssd_kernel_launches())


def test_set_forward_wait(wait_ns: int = 0, hold_unit: int = -1) -> None:
    """Test hook: bound on every device wait of the tensor-core forward (ns,
    0 = default) and a work unit that never publishes its state (-1 = none)."""
    load_library().ssd_test_set_forward_wait(int(wait_ns), int(hold_unit))


def test_set_backward_wait(polls: int = 0, hold: int = 0) -> None:
    """Test hook: bound on every mbarrier wait of the tensor-core backward
    (polls, 0 = default) and one MMA completion held back (1: gradient
    kernel, 2: state scan, 0: none)."""
    load_library().ssd_test_set_backward_wait(int(polls), int(hold))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SSD_DT_BF16
    if t.dtype == torch.float32:
        return SSD_DT_F32
    raise TypeError(f"x/dt/B/C must be bfloat16 or float32, got {t.dtype}")


def _need(t, name, device, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def ssd_chunk_scan_fwd_workspace_size(batch, seqlen, nheads, headdim, dstate, ngroups,
                                      chunk_size, in_dtype, varlen=False, nseq=0) -> int:
    n = load_library().ssd_chunk_scan_fwd_workspace_size(
        batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, in_dtype, int(bool(varlen)),
        nseq)
    if n == ctypes.c_size_t(-1).value:
        raise SSDError(SSD_ERR_UNSUPPORTED, "ssd_chunk_scan_fwd_workspace_size")
    return int(n)


def ssd_chunk_scan_fwd(x, dt, A, B, C, D=None, chunk_size=256, init_states=None,
                       cu_seqlens=None, *, y=None, final_states=None, return_final=True,
                       workspace=None, dev_status=None, stream=None, dt_bias=None,
                       dt_softplus=False, z=None, y_dtype=torch.float32):
    """SSD layer forward.  Shapes (device tensors, contiguous):

    x [b, T, H, P], dt [b, T, H], B/C [b, T, G, N] -- all bfloat16 or all
    float32; A [H] and D [H] float32; init_states [nseq_or_b, H, P, N]
    float32; cu_seqlens int32 [nseq + 1] (then b must be 1).

    Fused epilogue (ssd_chunk_scan_fwd_ex; tensor-core shapes only):
    ``dt_softplus`` uses softplus(dt + dt_bias) for dt (dt_bias [H] float32
    or None); ``z`` [b, T, H, P] multiplies y by silu(z); ``y_dtype``
    torch.bfloat16 writes y as bf16.

    Returns ``(y [b, T, H, P], final_states [nseq_or_b, H, P, N] float32 or
    None)``.  Raises SSDError on a host-side rejection.  Errors only the
    device can detect go to ``dev_status`` (an int32 device tensor of one
    element) when given.
    """
    lib = load_library()
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("ssd_chunk_scan_fwd needs CUDA tensors")
    if x.dim() != 4:
        raise ValueError("x must be [batch, seqlen, nheads, headdim]")
    b, T, H, P = x.shape
    if B.dim() != 4:
        raise ValueError("B must be [batch, seqlen, ngroups, dstate]")
    G, N = B.shape[2], B.shape[3]
    code = _dtype_code(x)
    _need(x, "x", dev)
    _need(dt, "dt", dev, x.dtype, (b, T, H))
    _need(B, "B", dev, x.dtype, (b, T, G, N))
    _need(C, "C", dev, x.dtype, (b, T, G, N))
    _need(A, "A", dev, torch.float32, (H,))
    if D is not None:
        _need(D, "D", dev, torch.float32, (H,))
    nseq = b
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", dev, torch.int32)
        nseq = cu_seqlens.shape[0] - 1
    if init_states is not None:
        _need(init_states, "init_states", dev, torch.float32, (nseq, H, P, N))
    if y_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("y_dtype must be torch.float32 or torch.bfloat16")
    if dt_bias is not None:
        _need(dt_bias, "dt_bias", dev, torch.float32, (H,))
    if z is not None:
        _need(z, "z", dev, x.dtype, (b, T, H, P))
    fused = bool(dt_softplus) or z is not None or y_dtype == torch.bfloat16
    if y is None:
        y = torch.empty((b, T, H, P), device=dev, dtype=y_dtype)
    _need(y, "y", dev, y_dtype, (b, T, H, P))
    if final_states is None and return_final:
        final_states = torch.empty((nseq, H, P, N), device=dev, dtype=torch.float32)
    if final_states is not None:
        _need(final_states, "final_states", dev, torch.float32, (nseq, H, P, N))
    need = ssd_chunk_scan_fwd_workspace_size(b, T, H, P, N, G, chunk_size, code,
                                             cu_seqlens is not None, nseq)
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if fused:
        epi = FwdEpilogue(None if dt_bias is None else dt_bias.data_ptr(), int(bool(dt_softplus)),
                          None if z is None else z.data_ptr(), int(y_dtype == torch.bfloat16))
        st = lib.ssd_chunk_scan_fwd_ex(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), b, T,
                                       H, P, N, G, chunk_size, code, _ptr(init_states),
                                       _ptr(cu_seqlens), nseq, _ptr(y), _ptr(final_states),
                                       _ptr(workspace), ws_bytes, _ptr(dev_status),
                                       _stream_handle(stream), ctypes.byref(epi))
        where = "ssd_chunk_scan_fwd_ex"
    else:
        st = lib.ssd_chunk_scan_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), b, T,
                                    H, P, N, G, chunk_size, code, _ptr(init_states),
                                    _ptr(cu_seqlens), nseq, _ptr(y), _ptr(final_states),
                                    _ptr(workspace), ws_bytes, _ptr(dev_status),
                                    _stream_handle(stream))
        where = "ssd_chunk_scan_fwd"
    if st != SSD_OK:
        raise SSDError(st, where)
    return y, final_states


def ssd_chunk_scan_states(x, dt, A, B, chunk_size=256, init_states=None, cu_seqlens=None, *,
                          final_states=None, workspace=None, dev_status=None, stream=None):
    """The state at the end of each sequence without the outputs
    (ssd_chunk_scan_states): shapes as for ``ssd_chunk_scan_fwd`` (no C, D,
    y).  Returns ``final_states [nseq_or_b, H, P, N]`` float32."""
    lib = load_library()
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("ssd_chunk_scan_states needs CUDA tensors")
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [batch, seqlen, nheads, headdim], B [batch, seqlen, ngroups, dstate]")
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    code = _dtype_code(x)
    _need(x, "x", dev)
    _need(dt, "dt", dev, x.dtype, (b, T, H))
    _need(B, "B", dev, x.dtype, (b, T, G, N))
    _need(A, "A", dev, torch.float32, (H,))
    nseq = b
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", dev, torch.int32)
        nseq = cu_seqlens.shape[0] - 1
    if init_states is not None:
        _need(init_states, "init_states", dev, torch.float32, (nseq, H, P, N))
    if final_states is None:
        final_states = torch.empty((nseq, H, P, N), device=dev, dtype=torch.float32)
    _need(final_states, "final_states", dev, torch.float32, (nseq, H, P, N))
    need = lib.ssd_chunk_scan_states_workspace_size(b, T, H, P, N, G, chunk_size, code,
                                                    int(cu_seqlens is not None), nseq)
    if need == ctypes.c_size_t(-1).value:
        raise SSDError(SSD_ERR_UNSUPPORTED, "ssd_chunk_scan_states_workspace_size")
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.ssd_chunk_scan_states(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), b, T, H, P, N, G,
                                   chunk_size, code, _ptr(init_states), _ptr(cu_seqlens), nseq,
                                   _ptr(final_states), _ptr(workspace), ws_bytes,
                                   _ptr(dev_status), _stream_handle(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_chunk_scan_states")
    return final_states


def ssd_state_update(state, x, dt, A, B, C, D=None, *, y=None, stream=None):
    """One decode step in place on ``state`` [b, H, P, N] float32.

    x [b, H, P], dt [b, H], B/C [b, G, N] (bfloat16 or float32); A, D [H]
    float32.  Returns y [b, H, P] float32.
    """
    lib = load_library()
    dev = state.device
    if dev.type != "cuda":
        raise ValueError("ssd_state_update needs CUDA tensors")
    b, H, P, N = state.shape
    G = B.shape[1]
    code = _dtype_code(x)
    _need(state, "state", dev, torch.float32)
    _need(x, "x", dev, None, (b, H, P))
    _need(dt, "dt", dev, x.dtype, (b, H))
    _need(B, "B", dev, x.dtype, (b, G, N))
    _need(C, "C", dev, x.dtype, (b, G, N))
    _need(A, "A", dev, torch.float32, (H,))
    if D is not None:
        _need(D, "D", dev, torch.float32, (H,))
    if y is None:
        y = torch.empty((b, H, P), device=dev, dtype=torch.float32)
    _need(y, "y", dev, torch.float32, (b, H, P))
    st = lib.ssd_state_update(_ptr(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                              b, H, P, N, G, code, _ptr(y), _stream_handle(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_state_update")
    return y


def ssd_selective_scan_fwd(x, dt, A, B, C, D=None, init_states=None, *, y=None,
                           final_states=None, return_final=True, stream=None):
    """Mamba-1 selective scan (a decay per channel and state).  Shapes
    (device tensors, contiguous):

    x, dt [b, L, Dm] and B, C [b, L, N] -- all bfloat16 or all float32;
    A [Dm, N], D [Dm] and init_states [b, Dm, N] float32.

    Returns ``(y [b, L, Dm] float32, final_states [b, Dm, N] float32 or
    None)``.  Raises SSDError on a host-side rejection.
    """
    lib = load_library()
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("ssd_selective_scan_fwd needs CUDA tensors")
    if x.dim() != 3 or A.dim() != 2:
        raise ValueError("x must be [batch, seqlen, dmodel] and A [dmodel, dstate]")
    b, L, Dm = x.shape
    N = A.shape[1]
    code = _dtype_code(x)
    _need(x, "x", dev)
    _need(dt, "dt", dev, x.dtype, (b, L, Dm))
    _need(B, "B", dev, x.dtype, (b, L, N))
    _need(C, "C", dev, x.dtype, (b, L, N))
    _need(A, "A", dev, torch.float32, (Dm, N))
    if D is not None:
        _need(D, "D", dev, torch.float32, (Dm,))
    if init_states is not None:
        _need(init_states, "init_states", dev, torch.float32, (b, Dm, N))
    if y is None:
        y = torch.empty((b, L, Dm), device=dev, dtype=torch.float32)
    _need(y, "y", dev, torch.float32, (b, L, Dm))
    if final_states is None and return_final:
        final_states = torch.empty((b, Dm, N), device=dev, dtype=torch.float32)
    if final_states is not None:
        _need(final_states, "final_states", dev, torch.float32, (b, Dm, N))
    st = lib.ssd_selective_scan_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                    _ptr(init_states), b, L, Dm, N, code, _ptr(y),
                                    _ptr(final_states), _stream_handle(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_selective_scan_fwd")
    return y, final_states


def ssd_segment_decay(dt, A, *, out=None, stream=None):
    """Total log-decay of a slice, A[h] * sum_t dt[b, t, h]: dt [b, T, H]
    (bfloat16 or float32), A [H] float32.  Returns [b, H] float32."""
    lib = load_library()
    dev = dt.device
    if dev.type != "cuda" or dt.dim() != 3:
        raise ValueError("dt must be a CUDA tensor [batch, seqlen, nheads]")
    b, T, H = dt.shape
    code = _dtype_code(dt)
    _need(dt, "dt", dev)
    _need(A, "A", dev, torch.float32, (H,))
    if out is None:
        out = torch.empty((b, H), device=dev, dtype=torch.float32)
    _need(out, "out", dev, torch.float32, (b, H))
    st = lib.ssd_segment_decay(_ptr(dt), _ptr(A), b, T, H, code, _ptr(out), _stream_handle(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_segment_decay")
    return out


def ssd_segment_combine(decay, states, init_states=None, *, out=None, stream=None):
    """States entering R consecutive slices: decay [R, b, H], states [R, b,
    H, P, N] (each slice's end state from a zero start), init_states [b, H,
    P, N] or None.  Returns [R + 1, b, H, P, N] float32: out[0] = init,
    out[r + 1] = exp(decay[r]) out[r] + states[r]."""
    lib = load_library()
    dev = states.device
    if dev.type != "cuda" or states.dim() != 5:
        raise ValueError("states must be a CUDA tensor [R, batch, nheads, headdim, dstate]")
    R, b, H, P, N = states.shape
    _need(states, "states", dev, torch.float32)
    _need(decay, "decay", dev, torch.float32, (R, b, H))
    if init_states is not None:
        _need(init_states, "init_states", dev, torch.float32, (b, H, P, N))
    if out is None:
        out = torch.empty((R + 1, b, H, P, N), device=dev, dtype=torch.float32)
    _need(out, "out", dev, torch.float32, (R + 1, b, H, P, N))
    st = lib.ssd_segment_combine(_ptr(decay), _ptr(states), _ptr(init_states), R, b, H, P, N,
                                 _ptr(out), _stream_handle(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_segment_combine")
    return out


def ssd_chunk_scan_bwd(x, dt, A, B, C, D, init_states, dy, dfinal=None, *, workspace=None,
                       want_dD=True, want_dinit=True, dev_status=None, stream=None):
    """Backward of the forward (batch mode).  x, dt, A, B, C, D, init_states
    as for ssd_chunk_scan_fwd; dy [b, T, H, P] float32; dfinal [b, H, P, N]
    float32 or None; dev_status an int32 device tensor (or None) that
    receives device-side errors.  Returns a dict of float32 gradients dx,
    ddt, dA, dB, dC and (unless disabled) dD and dinit."""
    lib = load_library()
    dev = x.device
    if dev.type != "cuda" or x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [b, T, H, P] and B [b, T, G, N], on a CUDA device")
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    code = _dtype_code(x)
    _need(x, "x", dev)
    _need(dt, "dt", dev, x.dtype, (b, T, H))
    _need(B, "B", dev, x.dtype, (b, T, G, N))
    _need(C, "C", dev, x.dtype, (b, T, G, N))
    _need(A, "A", dev, torch.float32, (H,))
    _need(dy, "dy", dev, torch.float32, (b, T, H, P))
    if D is not None:
        _need(D, "D", dev, torch.float32, (H,))
    if init_states is not None:
        _need(init_states, "init_states", dev, torch.float32, (b, H, P, N))
    if dfinal is not None:
        _need(dfinal, "dfinal", dev, torch.float32, (b, H, P, N))
    f32 = dict(device=dev, dtype=torch.float32)
    g = {"dx": torch.empty((b, T, H, P), **f32), "ddt": torch.empty((b, T, H), **f32),
         "dA": torch.empty((H,), **f32), "dB": torch.empty((b, T, G, N), **f32),
         "dC": torch.empty((b, T, G, N), **f32),
         "dD": torch.empty((H,), **f32) if want_dD else None,
         "dinit": torch.empty((b, H, P, N), **f32) if want_dinit else None}
    need = lib.ssd_chunk_scan_bwd_workspace_size(b, T, H, P, N, G, code)
    if need == ctypes.c_size_t(-1).value:
        raise SSDError(SSD_ERR_UNSUPPORTED, "ssd_chunk_scan_bwd_workspace_size")
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.ssd_chunk_scan_bwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), b, T, H, P,
                                N, G, code, _ptr(init_states), _ptr(dy), _ptr(dfinal),
                                _ptr(g["dx"]), _ptr(g["ddt"]), _ptr(g["dA"]), _ptr(g["dB"]),
                                _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["dinit"]), _ptr(workspace),
                                ws_bytes, _ptr(dev_status), _stream_handle(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_chunk_scan_bwd")
    return g
