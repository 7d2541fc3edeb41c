"""Pins of the backward oracle (CPU): every gradient against central finite
differences of the forward oracle, in fp64, on tiny inputs with two groups,
an initial state, D and a final-state cotangent.  The loss is
L = sum(y * dy) + sum(final * dfinal), so dL/dy = dy and dL/dfinal = dfinal."""
import numpy as np
import pytest

import oracle


def _inputs(seed, b=2, T=6, H=4, P=2, N=3, G=2):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((b, T, H, P)), dt=rng.uniform(0.05, 0.6, (b, T, H)),
                A=-rng.uniform(0.2, 2.0, H), B=rng.standard_normal((b, T, G, N)),
                C=rng.standard_normal((b, T, G, N)), D=rng.standard_normal(H),
                init=rng.standard_normal((b, H, P, N)))


def _loss(v, dy, dfin):
    y, fin = oracle.ssd_scan(v["x"], v["dt"], v["A"], v["B"], v["C"], v["D"], v["init"])
    return float(np.sum(y * dy) + np.sum(fin * dfin))


@pytest.mark.parametrize("seed", [1, 2])
def test_backward_matches_finite_differences(seed):
    v = _inputs(seed)
    rng = np.random.default_rng(100 + seed)
    b, T, H, P = v["x"].shape
    N = v["B"].shape[3]
    dy = rng.standard_normal((b, T, H, P))
    dfin = rng.standard_normal((b, H, P, N))
    g = oracle.ssd_bwd(v["x"], v["dt"], v["A"], v["B"], v["C"], v["D"], v["init"], dy, dfin)
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "init": "dinit"}
    eps = 1e-6
    for name, gname in names.items():
        fd = np.zeros_like(v[name])
        for idx in np.ndindex(v[name].shape):
            w = {k: a.copy() for k, a in v.items()}
            w[name][idx] += eps
            lp = _loss(w, dy, dfin)
            w[name][idx] -= 2 * eps
            lm = _loss(w, dy, dfin)
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.max(np.abs(g[gname] - fd)) / max(1e-12, np.max(np.abs(fd)))
        assert err < 1e-7, f"{gname}: relative error {err:.2e} against finite differences"


def test_backward_without_cotangent_of_the_final_state():
    v = _inputs(3, G=1)
    rng = np.random.default_rng(7)
    dy = rng.standard_normal(v["x"].shape)
    g0 = oracle.ssd_bwd(v["x"], v["dt"], v["A"], v["B"], v["C"], v["D"], v["init"], dy, None)
    g1 = oracle.ssd_bwd(v["x"], v["dt"], v["A"], v["B"], v["C"], v["D"], v["init"], dy,
                        np.zeros(v["init"].shape))
    for k in g0:
        np.testing.assert_array_equal(g0[k], g1[k])
