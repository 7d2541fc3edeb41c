"""Oracle for the SSD layer forward and the decode step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  The product path (the CUDA library and its
binding) never imports it, and this module imports nothing from the product.

Contents, all fp64:

* :func:`ssd_scan` / :func:`ssd_step` -- the definition: the token-by-token
  recurrence in plain C (``ssd_oracle.c``), loaded through ctypes.
* :func:`quadratic_form` -- the same map written as one materialised
  semiseparable matrix ``y = M x`` ("Transformers are SSMs Review",
  sec. 3-2 (1) and (2); "Mamba-2는 왜 Transformer와 닮았는가", section "SSD의
  핵심": recurrent, quadratic and matrix forms are one transformation).
* :func:`brute_force` -- a third coding: explicit products of the decays, no
  cumulative sums, pure Python loops, tiny inputs only.
* :func:`chunked_reference` -- the block decomposition the SSD algorithm
  uses ("Transformers are SSMs Review", sec. 3-2 (4)): intra-chunk quadratic
  blocks, per-chunk states, state passing between chunks, and the
  off-diagonal correction.  It is a second, independent statement of the same
  result, pinned against :func:`ssd_scan` in the tests.
* :func:`linear_attention` -- the A = 0 special case, causal linear attention
  as a masked matrix product ("Transformers are SSMs Review", sec. 3-2 (2)).
* :func:`softplus`, :func:`silu_gate` -- the elementwise steps either side
  of the layer in a Mamba block (positive step size, output gate), for the
  fused-epilogue options.
* :func:`ssd_bwd` -- the backward of the layer (reverse-mode, in C),
  pinned by finite differences of :func:`ssd_scan`.
* :func:`s6_scan` -- the Mamba-1 selective scan (a decay per channel and
  state), the sequential loop of "20.1 상태 공간 모델 (SSM)", sec. 5, in C;
  :func:`s6_brute_force` restates it with explicit products of the decays.

Readings shared by every function here (the pages leave them open): head h
uses group ``floor(h*G/H)``; ``D`` is one scalar per head; a missing initial
state is zero; ``y_t`` reads the state after token t's update.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c with gcc into libssd_oracle.so (next to it)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path):
    """Open a compiled oracle library and declare its two entry points."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    ci = ctypes.c_int
    lib.oracle_ssd_scan.argtypes = [dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, ci,
                                    dp, ip, ci, dp, dp, ci]
    lib.oracle_ssd_scan.restype = ci
    lib.oracle_ssd_step.argtypes = [dp, dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, dp]
    lib.oracle_ssd_step.restype = ci
    lib.oracle_s6_scan.argtypes = [dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, dp, dp, dp, ci]
    lib.oracle_s6_scan.restype = ci
    lib.oracle_ssd_bwd.argtypes = [dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, ci, dp, dp, dp,
                                   dp, dp, dp, dp, dp, dp, dp]
    lib.oracle_ssd_bwd.restype = ci
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB_PATH)
    return _lib


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def ssd_scan(x, dt, A, B, C, D=None, init=None, cu_seqlens=None, nthreads=None, lib=None):
    """Sequential fp64 recurrence.  Shapes:

    batch mode:  x [b,T,H,P], dt [b,T,H], B/C [b,T,G,N], init [b,H,P,N]
    varlen mode: same with b == 1 and ``cu_seqlens`` [S+1]; init [S,H,P,N]

    Returns ``(y [b,T,H,P], final [nseq,H,P,N])`` as float64 arrays.
    ``lib`` selects another build of the C source (the mutation tests use it).
    """
    lib = lib or _load()
    x, dt, A, B, C, D, init = map(_f64, (x, dt, A, B, C, D, init))
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dt.shape == (b, T, H) and A.shape == (H,)
    assert B.shape == (b, T, G, N) and C.shape == (b, T, G, N)
    cu = None
    if cu_seqlens is not None:
        assert b == 1
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        nseq = cu.shape[0] - 1
    else:
        nseq = b
    if D is not None:
        assert D.shape == (H,)
    if init is not None:
        assert init.shape == (nseq, H, P, N)
    y = np.empty((b, T, H, P), np.float64)
    final = np.empty((nseq, H, P, N), np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib.oracle_ssd_scan(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                             b, T, H, P, N, G, _ptr(init), _ptr(cu, ctypes.c_int32),
                             nseq, _ptr(y), _ptr(final), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_ssd_scan rejected its arguments (rc={rc})")
    return y, final


def ssd_step(state, x, dt, A, B, C, D=None, lib=None):
    """One decode step: returns ``(y [b,H,P], new_state [b,H,P,N])``.

    state [b,H,P,N], x [b,H,P], dt [b,H], B/C [b,G,N].  The input state is
    not modified.
    """
    lib = lib or _load()
    st = np.array(state, dtype=np.float64, copy=True, order="C")
    x, dt, A, B, C, D = map(_f64, (x, dt, A, B, C, D))
    b, H, P, N = st.shape
    G = B.shape[1]
    y = np.empty((b, H, P), np.float64)
    rc = lib.oracle_ssd_step(_ptr(st), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                             _ptr(D), b, H, P, N, G, _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_ssd_step rejected its arguments (rc={rc})")
    return y, st


def ssd_bwd(x, dt, A, B, C, D, init, dy, dfinal=None, lib=None):
    """Backward of the SSD layer, batch mode, fp64 (reverse-mode derivative
    of the recurrence of :func:`ssd_scan`, for dL/dy = dy and dL/dfinal =
    dfinal).  Returns a dict with dx, ddt, dA, dB, dC, dD, dinit, shaped like
    x, dt, A, B, C, A and the states."""
    lib = lib or _load()
    x, dt, A, B, C, D, init, dy, dfinal = map(_f64, (x, dt, A, B, C, D, init, dy, dfinal))
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    out = {"dx": np.empty_like(x), "ddt": np.empty_like(dt), "dA": np.empty(H),
           "dB": np.empty_like(B), "dC": np.empty_like(C), "dD": np.empty(H),
           "dinit": np.empty((b, H, P, N))}
    rc = lib.oracle_ssd_bwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), b, T, H, P, N, G,
                            _ptr(init), _ptr(dy), _ptr(dfinal), _ptr(out["dx"]), _ptr(out["ddt"]),
                            _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
                            _ptr(out["dinit"]))
    if rc != 0:
        raise ValueError(f"oracle_ssd_bwd rejected its arguments (rc={rc})")
    return out


def s6_scan(x, dt, A, B, C, D=None, init=None, nthreads=None, lib=None):
    """Mamba-1 selective scan, sequential fp64 loop.  Shapes:

    x, dt [b, L, Dm]; A [Dm, N]; B, C [b, L, N]; D [Dm]; init [b, Dm, N].
    Per channel d and state n: h = exp(dt_t[d] A[d,n]) h + dt_t[d] B_t[n] x_t[d],
    y_t[d] = sum_n h[n] C_t[n] + D[d] x_t[d].  Returns ``(y [b,L,Dm],
    final [b,Dm,N])`` as float64 arrays.
    """
    lib = lib or _load()
    x, dt, A, B, C, D, init = map(_f64, (x, dt, A, B, C, D, init))
    b, L, Dm = x.shape
    N = A.shape[1]
    assert dt.shape == (b, L, Dm) and A.shape == (Dm, N)
    assert B.shape == (b, L, N) and C.shape == (b, L, N)
    if D is not None:
        assert D.shape == (Dm,)
    if init is not None:
        assert init.shape == (b, Dm, N)
    y = np.empty((b, L, Dm), np.float64)
    final = np.empty((b, Dm, N), np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib.oracle_s6_scan(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), b, L, Dm, N,
                            _ptr(init), _ptr(y), _ptr(final), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_s6_scan rejected its arguments (rc={rc})")
    return y, final


def s6_brute_force(x, dt, A, B, C, D=None, init=None):
    """The selective scan written out, pure Python, tiny inputs only:

    y_i[d] = sum_n C_i[n] * ( sum_{j<=i} (prod_{k=j+1..i} exp(dt_k[d] A[d,n]))
                               * dt_j[d] B_j[n] x_j[d]
                              + (prod_{k<=i} exp(dt_k[d] A[d,n])) init[d,n] )
             + D[d] x_i[d]
    """
    import math
    x, dt, A, B, C, D, init = map(_f64, (x, dt, A, B, C, D, init))
    b, L, Dm = x.shape
    N = A.shape[1]
    y = np.zeros((b, L, Dm))
    for bi in range(b):
        for d in range(Dm):
            for i in range(L):
                acc = 0.0
                for n in range(N):
                    a = [math.exp(float(dt[bi, k, d]) * float(A[d, n])) for k in range(L)]
                    hn = 0.0
                    for j in range(i + 1):
                        dec = 1.0
                        for k in range(j + 1, i + 1):
                            dec *= a[k]
                        hn += dec * float(dt[bi, j, d]) * float(B[bi, j, n]) * float(x[bi, j, d])
                    if init is not None:
                        dec = 1.0
                        for k in range(i + 1):
                            dec *= a[k]
                        hn += dec * float(init[bi, d, n])
                    acc += float(C[bi, i, n]) * hn
                if D is not None:
                    acc += float(D[d]) * float(x[bi, i, d])
                y[bi, i, d] = acc
    return y


def _group_of(H, G):
    return [(h * G) // H for h in range(H)]


def quadratic_form(x, dt, A, B, C, D=None, init=None):
    """Materialised semiseparable matrix, one sequence per batch row.

    For j <= i:  M[i, j] = (C_i . B_j) * exp(sum_{k=j+1..i} dt_k A) * dt_j
    plus the initial-state term  C_i . (exp(sum_{k<=i} dt_k A) * init)  and
    the skip term D x_i.  O(T^2) memory: small inputs only.
    """
    x, dt, A, B, C, D, init = map(_f64, (x, dt, A, B, C, D, init))
    b, T, H, P = x.shape
    G = B.shape[2]
    grp = _group_of(H, G)
    y = np.zeros((b, T, H, P))
    final = np.zeros((b, H, P, B.shape[3]))
    for bi in range(b):
        for h in range(H):
            g = grp[h]
            la = dt[bi, :, h] * A[h]                    # log a_t
            cs = np.cumsum(la)                           # sum_{k<=i} log a_k
            seg = cs[:, None] - cs[None, :]              # sum_{k=j+1..i}
            causal = np.tril(np.ones((T, T), dtype=bool))
            L = np.where(causal, np.exp(np.where(causal, seg, 0.0)), 0.0)
            CB = C[bi, :, g, :] @ B[bi, :, g, :].T       # [T, T]
            M = CB * L * dt[bi, None, :, h]
            y[bi, :, h, :] = M @ x[bi, :, h, :]
            if init is not None:
                # y_init[i, p] = exp(cs_i) * sum_n C[i, n] init[p, n]
                y[bi, :, h, :] += np.exp(cs)[:, None] * (C[bi, :, g, :] @ init[bi, h].T)
            if D is not None:
                y[bi, :, h, :] += D[h] * x[bi, :, h, :]
            # final state from the same matrix view: last row of the decays
            w = np.exp(cs[-1] - cs) * dt[bi, :, h]       # weight of token j in h_T
            fin = (x[bi, :, h, :] * w[:, None]).T @ B[bi, :, g, :]
            if init is not None:
                fin += np.exp(cs[-1]) * init[bi, h]
            final[bi, h] = fin
    return y, final


def brute_force(x, dt, A, B, C, D=None, init=None):
    """Pure-Python loops with explicit products of the decays.

    y_i = sum_{j<=i} (prod_{k=j+1..i} a_k) * dt_j * x_j * (C_i . B_j)
          + (prod_{k<=i} a_k) * C_i . init + D x_i,  a_k = exp(dt_k A).
    Tiny inputs only (T <= ~16, P, N <= ~4).
    """
    x, dt, A, B, C, D, init = map(_f64, (x, dt, A, B, C, D, init))
    import math
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    grp = _group_of(H, G)
    y = np.zeros((b, T, H, P))
    for bi in range(b):
        for h in range(H):
            g = grp[h]
            a = [math.exp(float(dt[bi, t, h]) * float(A[h])) for t in range(T)]
            for i in range(T):
                for p in range(P):
                    acc = 0.0
                    for j in range(i + 1):
                        dec = 1.0
                        for k in range(j + 1, i + 1):
                            dec *= a[k]
                        cb = 0.0
                        for n in range(N):
                            cb += float(C[bi, i, g, n]) * float(B[bi, j, g, n])
                        acc += dec * float(dt[bi, j, h]) * float(x[bi, j, h, p]) * cb
                    if init is not None:
                        dec = 1.0
                        for k in range(i + 1):
                            dec *= a[k]
                        ch = 0.0
                        for n in range(N):
                            ch += float(C[bi, i, g, n]) * float(init[bi, h, p, n])
                        acc += dec * ch
                    if D is not None:
                        acc += float(D[h]) * float(x[bi, i, h, p])
                    y[bi, i, h, p] = acc
    return y


def chunked_reference(x, dt, A, B, C, D=None, init=None, chunk=64):
    """The SSD block decomposition in fp64, for any chunk length Q >= 1.

    Per sequence and head, with chunks c of length Q (the last may be short),
    cum_i = sum of dt_k A over the chunk up to and including i:

      1. intra-chunk (diagonal block):  Y_diag = (C B^T o L o dt_j) X,
         L[i, j] = exp(cum_i - cum_j) for j <= i, else 0;
      2. chunk state:  S_c = sum_j exp(cum_last - cum_j) dt_j x_j B_j^T;
      3. state passing:  H_c = exp(cum_last) H_{c-1} + S_c, H_{-1} = init;
      4. off-diagonal output:  Y_off[i] = exp(cum_i) C_i H_{c-1}^T;
      y = Y_diag + Y_off + D x.

    Returns ``(y, final)`` like :func:`ssd_scan` in batch mode.
    """
    x, dt, A, B, C, D, init = map(_f64, (x, dt, A, B, C, D, init))
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    grp = _group_of(H, G)
    y = np.zeros((b, T, H, P))
    final = np.zeros((b, H, P, N))
    for bi in range(b):
        for h in range(H):
            g = grp[h]
            state = np.zeros((P, N)) if init is None else init[bi, h].copy()
            for c0 in range(0, T, chunk):
                c1 = min(T, c0 + chunk)
                X = x[bi, c0:c1, h, :]
                Bc = B[bi, c0:c1, g, :]
                Cc = C[bi, c0:c1, g, :]
                d = dt[bi, c0:c1, h]
                cum = np.cumsum(d * A[h])
                q = c1 - c0
                causal = np.tril(np.ones((q, q), dtype=bool))
                L = np.where(causal, np.exp(np.where(causal, cum[:, None] - cum[None, :], 0.0)), 0.0)
                Yd = ((Cc @ Bc.T) * L * d[None, :]) @ X                       # step 1
                Sc = (X * (np.exp(cum[-1] - cum) * d)[:, None]).T @ Bc         # step 2
                Yo = np.exp(cum)[:, None] * (Cc @ state.T)                     # step 4
                state = np.exp(cum[-1]) * state + Sc                           # step 3
                y[bi, c0:c1, h, :] = Yd + Yo
            if D is not None:
                y[bi, :, h, :] += D[h] * x[bi, :, h, :]
            final[bi, h] = state
    return y, final


def linear_attention(x, dt, B, C):
    """Causal linear attention, y_i = sum_{j<=i} (C_i . B_j) dt_j x_j.

    Written as a masked matrix product: tril(C B^T diag(dt)) X.  This is
    what the selective recurrence reduces to when A = 0 (no decay), with a
    zero initial state and no skip term.
    """
    x, dt, B, C = map(_f64, (x, dt, B, C))
    b, T, H, P = x.shape
    G = B.shape[2]
    grp = _group_of(H, G)
    y = np.zeros((b, T, H, P))
    for bi in range(b):
        for h in range(H):
            g = grp[h]
            Wm = np.tril(C[bi, :, g, :] @ B[bi, :, g, :].T) * dt[bi, None, :, h]
            y[bi, :, h, :] = Wm @ x[bi, :, h, :]
    return y


def softplus(v):
    """softplus(v) = log(1 + exp(v)), fp64: the step size of the selective SSM
    is a softplus of a projection, which keeps it positive ("20.1 상태 공간
    모델 (SSM)", sec. 2, and the same page's sec. 5 loop)."""
    return np.logaddexp(0.0, np.asarray(v, dtype=np.float64))


def silu_gate(y, z):
    """y * silu(z), silu(z) = z / (1 + exp(-z)), fp64: the Mamba block's
    second branch is a gate multiplied into the SSM output (the Mamba paper
    review, sec. 5).  The page does not name the gate's nonlinearity; SiLU
    is the reading taken.  exp(-z) overflowing to inf gives the correct limit
    0 for very negative z."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return np.asarray(y, dtype=np.float64) * (z / (1.0 + np.exp(-z)))


def rel_err(got, ref):
    """max |got - ref| / RMS(ref): the tolerance metric used by the tests."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    diff = float(np.max(np.abs(got - ref)))
    return diff / rms if rms > 0 else diff
