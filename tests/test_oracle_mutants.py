"""The oracle's pins must catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, a wrong index, swapped operands), builds it with gcc in a
temporary directory, and runs the pin checks against it.  At least one pin
must fail for every mutant; the unmodified source must pass all of them.
"""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle import oracle as O

SRC = os.path.join(os.path.dirname(O.__file__), "ssd_oracle.c")

MUTANTS = {
    "drop_skip_term": ("yt[p] = acc + Dh * xt[p];", "yt[p] = acc;"),
    "decay_sign": ("const double a = exp(dtt * Ah);", "const double a = exp(-dtt * Ah);"),
    "drop_dt_on_input": ("const double u = dtt * xt[p];", "const double u = xt[p];"),
    "swap_B_C_in_update": ("hp[n] = a * hp[n] + u * Bt[n];", "hp[n] = a * hp[n] + u * Ct[n];"),
    "group_index_modulo": ("const int g = (int)(((int64_t)h * G) / H);\n    const double Ah",
                           "const int g = h % G;\n    const double Ah"),
    "y_before_update": ("                hp[n] = a * hp[n] + u * Bt[n];\n                acc += Ct[n] * hp[n];",
                        "                acc += Ct[n] * hp[n];\n                hp[n] = a * hp[n] + u * Bt[n];"),
    "init_index_transposed": ("memcpy(state, J->init + ((size_t)s * H + h) * PN",
                              "memcpy(state, J->init + ((size_t)h * J->nseq + s) * PN"),
    "decode_decay_missing": ("*e = a * *e + dtt * xt[p] * Bt[n];", "*e = *e + dtt * xt[p] * Bt[n];"),
    # the selective scan (a decay per channel and state)
    "s6_decay_of_state_0": ("const double dA = exp(dtt * Ad[n]);", "const double dA = exp(dtt * Ad[0]);"),
    "s6_A_transposed": ("const double dA = exp(dtt * Ad[n]);",
                        "const double dA = exp(dtt * J->A[(size_t)n * Dm + d]);"),
    "s6_drop_dt_on_input": ("h[n] = dA * h[n] + dtt * Bt[n] * xt;", "h[n] = dA * h[n] + Bt[n] * xt;"),
    "s6_y_before_update": ("                h[n] = dA * h[n] + dtt * Bt[n] * xt;\n                acc += h[n] * Ct[n];",
                           "                acc += h[n] * Ct[n];\n                h[n] = dA * h[n] + dtt * Bt[n] * xt;"),
    "s6_drop_skip_term": ("J->y[bt * Dm + d] = acc + Dd * xt;", "J->y[bt * Dm + d] = acc;"),
    "s6_init_ignored": ("h[n] = J->init ? J->init[((size_t)b * Dm + d) * N + n] : 0.0;", "h[n] = 0.0;"),
    # the backward
    "bwd_adjoint_not_decayed": ("for (size_t e = 0; e < PN; ++e) Gs[e] *= a;", "for (size_t e = 0; e < PN; ++e) Gs[e] *= 1.0;"),
    "bwd_dA_uses_h_t": ("s_h += gv * hp[p * N + n];", "s_h += gv * ht[p * N + n];"),
    "bwd_dC_uses_h_prev": ("gc += dyt[p] * ht[p * N + n];", "gc += dyt[p] * hp[p * N + n];"),
    "bwd_dx_drops_dt": ("dx[(bt * H + h) * P + p] = dtt * acc + Dh * dyt[p];", "dx[(bt * H + h) * P + p] = acc + Dh * dyt[p];"),
}


def _build(tmp_path, name, src_text):
    d = tmp_path / name
    d.mkdir()
    c = d / "m.c"
    c.write_text(src_text)
    so = d / "m.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           str(c), "-o", str(so), "-lm"])
    return O.load_library(str(so))


def _pins(lib):
    """Return the names of the pins this library fails."""
    failed = []
    rng = np.random.default_rng(21)
    # scalar-gate worked example (feghi.github.io review, sec. 3)
    for g, want in ((0.1, 9.2), (0.9, 2.8)):
        dt = -math.log(1 - g)
        y, _ = oracle.ssd_scan(np.full((1, 1, 1, 1), 2.0), np.full((1, 1, 1), dt), np.array([-1.0]),
                               np.full((1, 1, 1, 1), g / dt), np.ones((1, 1, 1, 1)), np.zeros(1),
                               np.full((1, 1, 1, 1), 10.0), lib=lib)
        if abs(y[0, 0, 0, 0] - want) > 1e-12:
            failed.append("scalar_gate")
            break
    # materialised semiseparable matrix, with init, D and 2 groups
    b, T, H, P, N, G = 2, 13, 4, 3, 4, 2
    x = rng.standard_normal((b, T, H, P))
    dt = rng.uniform(0.01, 0.5, (b, T, H))
    A = -rng.uniform(0.1, 2, H)
    B = rng.standard_normal((b, T, G, N))
    C = rng.standard_normal((b, T, G, N))
    D = rng.standard_normal(H)
    h0 = rng.standard_normal((b, H, P, N))
    y, fin = oracle.ssd_scan(x, dt, A, B, C, D, h0, lib=lib)
    yq, fq = oracle.quadratic_form(x, dt, A, B, C, D, h0)
    if oracle.rel_err(y, yq) > 1e-12 or oracle.rel_err(fin, fq) > 1e-12:
        failed.append("quadratic_form")
    # decode steps vs the materialised form
    st = h0.copy()
    for t in range(T):
        yt, st = oracle.ssd_step(st, x[:, t], dt[:, t], A, B[:, t], C[:, t], D, lib=lib)
        if oracle.rel_err(yt, yq[:, t]) > 1e-12:
            failed.append("decode_vs_quadratic")
            break
    # selective scan vs its explicit-products restatement (distinct A per
    # channel and state, Dm != N so a transposed A reads other values)
    b6, L6, Dm, N6 = 2, 7, 3, 4
    x6 = rng.standard_normal((b6, L6, Dm))
    dt6 = rng.uniform(0.05, 0.6, (b6, L6, Dm))
    A6 = -rng.uniform(0.2, 3.0, (Dm, N6))
    B6 = rng.standard_normal((b6, L6, N6))
    C6 = rng.standard_normal((b6, L6, N6))
    D6 = rng.standard_normal(Dm)
    i6 = rng.standard_normal((b6, Dm, N6))
    y6, _ = oracle.s6_scan(x6, dt6, A6, B6, C6, D6, i6, lib=lib)
    if oracle.rel_err(y6, oracle.s6_brute_force(x6, dt6, A6, B6, C6, D6, i6)) > 1e-12:
        failed.append("s6_explicit_products")
    # backward: each gradient against a directional central difference of the
    # forward, L = sum(y dy) + sum(final dfinal)
    b, T, H, P, N, G = 2, 5, 4, 2, 3, 2
    v = dict(x=rng.standard_normal((b, T, H, P)), dt=rng.uniform(0.05, 0.6, (b, T, H)),
             A=-rng.uniform(0.2, 2.0, H), B=rng.standard_normal((b, T, G, N)),
             C=rng.standard_normal((b, T, G, N)), D=rng.standard_normal(H),
             init=rng.standard_normal((b, H, P, N)))
    dy = rng.standard_normal((b, T, H, P))
    dfin = rng.standard_normal((b, H, P, N))

    def loss(w):
        yy, ff = oracle.ssd_scan(w["x"], w["dt"], w["A"], w["B"], w["C"], w["D"], w["init"], lib=lib)
        return float(np.sum(yy * dy) + np.sum(ff * dfin))

    gr = oracle.ssd_bwd(v["x"], v["dt"], v["A"], v["B"], v["C"], v["D"], v["init"], dy, dfin, lib=lib)
    for name, gname in (("x", "dx"), ("dt", "ddt"), ("A", "dA"), ("B", "dB"), ("C", "dC"),
                        ("D", "dD"), ("init", "dinit")):
        d = rng.standard_normal(v[name].shape)
        wp = {k: a.copy() for k, a in v.items()}
        wm = {k: a.copy() for k, a in v.items()}
        wp[name] += 1e-6 * d
        wm[name] -= 1e-6 * d
        fd = (loss(wp) - loss(wm)) / 2e-6
        if abs(float(np.sum(gr[gname] * d)) - fd) > 1e-6 * max(1.0, abs(fd)):
            failed.append(f"bwd_{gname}")
            break
    return failed


def test_unmodified_oracle_passes_all_pins(tmp_path):
    lib = _build(tmp_path, "orig", open(SRC).read())
    assert _pins(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    lib = _build(tmp_path, name, text.replace(old, new))
    assert _pins(lib), f"no pin caught mutant {name}"
