"""Pins of the Mamba-1 selective-scan oracle (CPU only).

The scan is the sequential loop of "20.1 상태 공간 모델 (SSM)"
(sungeuns.github.io), sec. 5: a decay exp(dt_t[d] A[d, n]) per channel d and
state n, input term dt_t[d] B_t[n] x_t[d], output sum_n h[n] C_t[n] + D[d]
x_t[d].  Each test checks the C oracle against something other than itself:
the SSD oracle on the inputs where the two layers coincide, a pure-Python
restatement with explicit products of the decays, closed forms, and
symmetries of the definition.
"""
import numpy as np

import oracle


def _inputs(rng, b, L, Dm, N, init=True, D=True):
    x = rng.standard_normal((b, L, Dm))
    dt = rng.uniform(0.01, 0.6, (b, L, Dm))
    A = -np.exp(rng.uniform(np.log(0.2), np.log(4.0), (Dm, N)))
    B = rng.standard_normal((b, L, N))
    C = rng.standard_normal((b, L, N))
    Dv = rng.standard_normal(Dm) if D else None
    h0 = rng.standard_normal((b, Dm, N)) if init else None
    return x, dt, A, B, C, Dv, h0


def test_s6_reduces_to_ssd_when_the_decay_is_shared():
    # SSD with one group is the selective scan whose channels d = (h, p) share
    # their head's dt and A across all states ("Transformers are SSMs
    # Review", sec. 3-2 (3): scalar-times-identity A).  The SSD oracle is a
    # separate code path, pinned on its own.
    rng = np.random.default_rng(5)
    b, T, H, P, N = 2, 37, 3, 4, 5
    x = rng.standard_normal((b, T, H, P))
    dt = rng.uniform(0.01, 0.5, (b, T, H))
    A = -rng.uniform(0.1, 3.0, H)
    B = rng.standard_normal((b, T, 1, N))
    C = rng.standard_normal((b, T, 1, N))
    D = rng.standard_normal(H)
    h0 = rng.standard_normal((b, H, P, N))
    ys, fs = oracle.ssd_scan(x, dt, A, B, C, D, h0)
    y6, f6 = oracle.s6_scan(x.reshape(b, T, H * P), np.repeat(dt, P, axis=2),
                            np.repeat(A, P)[:, None] * np.ones((1, N)), B[:, :, 0], C[:, :, 0],
                            np.repeat(D, P), h0.reshape(b, H * P, N))
    assert oracle.rel_err(y6, ys.reshape(b, T, H * P)) < 1e-13
    assert oracle.rel_err(f6, fs.reshape(b, H * P, N)) < 1e-13


def test_s6_matches_explicit_decay_products():
    rng = np.random.default_rng(11)
    x, dt, A, B, C, D, h0 = _inputs(rng, 2, 9, 3, 4)
    y, _ = oracle.s6_scan(x, dt, A, B, C, D, h0)
    assert oracle.rel_err(y, oracle.s6_brute_force(x, dt, A, B, C, D, h0)) < 1e-13
    y, _ = oracle.s6_scan(x, dt, A, B, C)
    assert oracle.rel_err(y, oracle.s6_brute_force(x, dt, A, B, C)) < 1e-13


def test_s6_zero_decay_is_a_running_sum():
    # A = 0: exp(0) = 1, the state is the running sum of dt B x
    rng = np.random.default_rng(3)
    x, dt, _, B, C, D, _ = _inputs(rng, 1, 50, 6, 8, init=False)
    A = np.zeros((6, 8))
    y, fin = oracle.s6_scan(x, dt, A, B, C, D)
    h = np.cumsum((dt * x)[:, :, :, None] * B[:, :, None, :], axis=1)    # [b, L, Dm, N]
    want = np.einsum("bldn,bln->bld", h, C) + D * x
    assert oracle.rel_err(y, want) < 1e-12
    assert oracle.rel_err(fin, h[:, -1]) < 1e-12


def test_s6_constant_input_reaches_the_geometric_fixed_point():
    # constant dt, x, B, C: h_t -> dt B x / (1 - exp(dt A)), per (d, n)
    Dm, N, L = 3, 4, 3000
    A = -np.array([[0.5, 1.0, 2.0, 4.0], [0.1, 0.3, 0.7, 1.3], [3.0, 2.0, 1.0, 0.25]])
    dtv, xv = 0.2, np.array([1.5, -0.5, 2.0])
    Bv, Cv = np.array([1.0, -2.0, 0.5, 3.0]), np.array([0.25, 1.0, -1.0, 2.0])
    x = np.broadcast_to(xv, (1, L, Dm)).copy()
    dt = np.full((1, L, Dm), dtv)
    B = np.broadcast_to(Bv, (1, L, N)).copy()
    C = np.broadcast_to(Cv, (1, L, N)).copy()
    D = np.array([0.5, -1.0, 2.0])
    y, fin = oracle.s6_scan(x, dt, A, B, C, D)
    h_inf = dtv * Bv[None, :] * xv[:, None] / (1.0 - np.exp(dtv * A))
    assert np.allclose(fin[0], h_inf, rtol=1e-12, atol=0)
    assert np.allclose(y[0, -1], h_inf @ Cv + D * xv, rtol=1e-12, atol=0)


def test_s6_state_and_channel_permutations():
    # the states of a channel are independent recurrences summed by C, and the
    # channels are independent: relabelling states leaves y unchanged,
    # relabelling channels relabels y
    rng = np.random.default_rng(8)
    x, dt, A, B, C, D, h0 = _inputs(rng, 2, 21, 5, 6)
    y, fin = oracle.s6_scan(x, dt, A, B, C, D, h0)
    pn = rng.permutation(6)
    y2, fin2 = oracle.s6_scan(x, dt, A[:, pn], B[:, :, pn], C[:, :, pn], D, h0[:, :, pn])
    assert oracle.rel_err(y2, y) < 1e-13 and oracle.rel_err(fin2, fin[:, :, pn]) < 1e-13
    pd = rng.permutation(5)
    y3, fin3 = oracle.s6_scan(x[:, :, pd], dt[:, :, pd], A[pd], B, C, D[pd], h0[:, pd])
    assert oracle.rel_err(y3, y[:, :, pd]) < 1e-13 and oracle.rel_err(fin3, fin[:, pd]) < 1e-13


def test_s6_pages_usage_shapes():
    # the usage example of the same section: batch 2, 128 steps, d_model 512,
    # d_state 16, A = -exp(A_log) with A_log ~ N(0, 1), dt > 0
    rng = np.random.default_rng(0)
    b, L, Dm, N = 2, 128, 512, 16
    x = rng.standard_normal((b, L, Dm))
    dt = np.log1p(np.exp(rng.standard_normal((b, L, Dm))))      # softplus
    A = -np.exp(rng.standard_normal((Dm, N)))
    B = rng.standard_normal((b, L, N))
    C = rng.standard_normal((b, L, N))
    D = rng.standard_normal(Dm)
    y, fin = oracle.s6_scan(x, dt, A, B, C, D)
    assert y.shape == (b, L, Dm) and fin.shape == (b, Dm, N)
    assert np.isfinite(y).all() and np.isfinite(fin).all()
