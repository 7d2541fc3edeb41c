"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: the pages'
worked example, a closed form, a textbook special case, an independent coding
(materialised matrix, brute force, block decomposition), or an invariant the
pages state.
"""
import math
import os

import numpy as np
import pytest

import oracle
from state_space_sequence_05_b300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(seed, b=2, T=23, H=4, P=3, N=5, G=2, init=True, D=True, amax=2.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((b, T, H, P))
    dt = rng.uniform(0.01, 0.5, (b, T, H))
    A = -rng.uniform(0.1, amax, H)
    B = rng.standard_normal((b, T, G, N))
    C = rng.standard_normal((b, T, G, N))
    Dv = rng.standard_normal(H) if D else None
    h0 = rng.standard_normal((b, H, P, N)) if init else None
    return x, dt, A, B, C, Dv, h0


def test_scalar_gate_worked_example():
    """feghi.github.io review, sec. 3: h = (1-g)*10 + g*2 -> 9.2 / 2.8.

    Mapping onto the layer: H=P=N=G=1, one token, A=-1, dt=-ln(1-g) so that
    exp(dt*A) = 1-g, B = g/dt so that dt*B*x = g*x, C=1, D=0, init = h_prev.
    """
    rows = [l.split() for l in open(os.path.join(GOLDEN, "scalar_gate.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    for g, h_prev, xv, h_new in (map(float, r) for r in rows):
        dt = -math.log(1.0 - g)
        x = np.full((1, 1, 1, 1), xv)
        y, fin = oracle.ssd_scan(x, np.full((1, 1, 1), dt), np.array([-1.0]),
                                 np.full((1, 1, 1, 1), g / dt), np.ones((1, 1, 1, 1)),
                                 np.zeros(1), np.full((1, 1, 1, 1), h_prev))
        assert abs(y[0, 0, 0, 0] - h_new) < 1e-12
        assert abs(fin[0, 0, 0, 0] - h_new) < 1e-12
        # the decode step is one iteration of the same loop
        ys, st = oracle.ssd_step(np.full((1, 1, 1, 1), h_prev), np.full((1, 1, 1), xv),
                                 np.full((1, 1), dt), np.array([-1.0]),
                                 np.full((1, 1, 1), g / dt), np.ones((1, 1, 1)), None)
        assert abs(ys[0, 0, 0] - h_new) < 1e-12 and abs(st[0, 0, 0, 0] - h_new) < 1e-12


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_materialised_semiseparable_matrix(seed):
    x, dt, A, B, C, D, h0 = _rand_problem(seed)
    y, fin = oracle.ssd_scan(x, dt, A, B, C, D, h0)
    yq, finq = oracle.quadratic_form(x, dt, A, B, C, D, h0)
    assert np.max(np.abs(y - yq)) <= 1e-12 * max(1.0, np.max(np.abs(yq)))
    assert np.max(np.abs(fin - finq)) <= 1e-12 * max(1.0, np.max(np.abs(finq)))


@pytest.mark.parametrize("seed", [3, 4])
def test_matches_brute_force_products(seed):
    x, dt, A, B, C, D, h0 = _rand_problem(seed, b=1, T=11, H=2, P=2, N=3, G=1)
    y, _ = oracle.ssd_scan(x, dt, A, B, C, D, h0)
    yb = oracle.brute_force(x, dt, A, B, C, D, h0)
    assert np.max(np.abs(y - yb)) <= 1e-12 * max(1.0, np.max(np.abs(yb)))


def test_A_zero_is_causal_linear_attention():
    """No decay: the layer is causal linear attention tril(C B^T diag(dt)) X."""
    x, dt, A, B, C, _, _ = _rand_problem(5, T=40, init=False, D=False)
    y, _ = oracle.ssd_scan(x, dt, np.zeros_like(A), B, C)
    yl = oracle.linear_attention(x, dt, B, C)
    assert np.max(np.abs(y - yl)) <= 1e-12 * np.max(np.abs(yl))


def test_dt_zero_freezes_state():
    """dt = 0: exp(0*A) = 1 and no input is written, so h stays at init and
    y = C . h_prev + D x ("20.1 상태 공간 모델 (SSM)", sec. 2: small step
    freezes the state)."""
    x, _, A, B, C, D, h0 = _rand_problem(6, T=9)
    dt = np.zeros(x.shape[:3])
    y, fin = oracle.ssd_scan(x, dt, A, B, C, D, h0)
    assert np.array_equal(fin, h0)
    H = x.shape[2]
    G = B.shape[2]
    for h in range(H):
        g = h * G // H
        want = np.einsum("btn,bpn->btp", C[:, :, g, :], h0[:, h]) + D[h] * x[:, :, h, :]
        assert np.max(np.abs(y[:, :, h, :] - want)) < 1e-12


def test_geometric_series_closed_form():
    """Constant a = exp(dt*A), B = C = 1, x = c, zero init, P = N = 1:
    h_t = dt*c*(1 - a^t)/(1 - a) after t tokens."""
    T, dtv, Av, c = 50, 0.3, -0.7, 1.7
    y, fin = oracle.ssd_scan(np.full((1, T, 1, 1), c), np.full((1, T, 1), dtv), np.array([Av]),
                             np.ones((1, T, 1, 1)), np.ones((1, T, 1, 1)))
    a = math.exp(dtv * Av)
    t = np.arange(1, T + 1)
    want = dtv * c * (1 - a ** t) / (1 - a)
    assert np.max(np.abs(y[0, :, 0, 0] - want)) < 1e-12
    assert abs(fin[0, 0, 0, 0] - want[-1]) < 1e-12


def _page4_selective_scan(x, dt, A_full, Bm, Cm, Dv):
    """The per-channel selective scan of "20.1 상태 공간 모델 (SSM)", sec. 5,
    restated: A has one value per (channel, state); for each token
    h <- exp(dt*A) * h + dt * B * x, then y = sum_n h * C + D * x."""
    b, T, Dm = x.shape
    N = A_full.shape[1]
    h = np.zeros((b, Dm, N))
    y = np.zeros_like(x)
    for t in range(T):
        decay = np.exp(dt[:, t, :, None] * A_full[None])
        h = decay * h + (dt[:, t, :, None] * Bm[:, t, None, :]) * x[:, t, :, None]
        y[:, t, :] = np.einsum("bdn,bn->bd", h, Cm[:, t, :]) + Dv[None, :] * x[:, t, :]
    return y


def test_page4_loop_special_case():
    """With A constant along d_state, the page's per-channel scan is the SSD
    layer with one head per channel, headdim 1 and one group.  Shapes as the
    page's usage example (batch 2, 128 tokens, d_model 512, d_state 16), whose
    only printed output is the shape [2, 128, 512]."""
    rng = np.random.default_rng(8)
    b, T, Dm, N = 2, 128, 512, 16
    x = rng.standard_normal((b, T, Dm))
    dt = np.log1p(np.exp(rng.standard_normal((b, T, Dm))))  # softplus, positive
    a_row = -np.exp(rng.standard_normal(Dm))
    A_full = np.repeat(a_row[:, None], N, axis=1)
    Bm = rng.standard_normal((b, T, N))
    Cm = rng.standard_normal((b, T, N))
    Dv = rng.standard_normal(Dm)
    want = _page4_selective_scan(x, dt, A_full, Bm, Cm, Dv)
    y, _ = oracle.ssd_scan(x[..., None], dt, a_row, Bm[:, :, None, :], Cm[:, :, None, :], Dv)
    assert y[..., 0].shape == (2, 128, 512)
    assert np.max(np.abs(y[..., 0] - want)) <= 1e-12 * np.max(np.abs(want))


@pytest.mark.parametrize("Q", [1, 2, 7, 64, 300])
def test_block_decomposition_equals_recurrence(Q):
    """The SSD chunked algorithm is an exact reordering: any chunk length
    gives the recurrence's result ("Transformers are SSMs Review", 3-2 (4))."""
    x, dt, A, B, C, D, h0 = _rand_problem(9, b=2, T=150, H=4, P=4, N=6, G=2)
    y, fin = oracle.ssd_scan(x, dt, A, B, C, D, h0)
    yc, finc = oracle.chunked_reference(x, dt, A, B, C, D, h0, chunk=Q)
    assert oracle.rel_err(yc, y) < 1e-12
    assert oracle.rel_err(finc, fin) < 1e-12


@pytest.mark.parametrize("k", [0, 1, 17, 40])
def test_state_carry_split(k):
    """Run [0,T) == run [0,k) then [k,T) with init = the first run's final
    state (sequence parallelism passes only boundary states, 3-2 (6))."""
    x, dt, A, B, C, D, h0 = _rand_problem(10, T=40)
    y, fin = oracle.ssd_scan(x, dt, A, B, C, D, h0)
    y1, f1 = oracle.ssd_scan(x[:, :k], dt[:, :k], A, B[:, :k], C[:, :k], D, h0)
    y2, f2 = oracle.ssd_scan(x[:, k:], dt[:, k:], A, B[:, k:], C[:, k:], D, f1)
    assert np.max(np.abs(np.concatenate([y1, y2], 1) - y)) < 1e-12
    assert np.max(np.abs(f2 - fin)) < 1e-12


def test_final_state_is_affine_in_init_and_composes():
    """Each token applies h -> a h + b.  Composition (a2,b2)o(a1,b1) =
    (a2 a1, a2 b1 + b2) is associative but not commutative (feghi.github.io
    review, sec. 4).  Check: final(init) = (prod a) init + final(0), and the
    segment maps of two halves compose to the map of the whole."""
    x, dt, A, B, C, D, h0 = _rand_problem(11, b=1, T=30, H=2, G=1)
    _, f0 = oracle.ssd_scan(x, dt, A, B, C, D, None)
    _, fi = oracle.ssd_scan(x, dt, A, B, C, D, h0)
    prod_a = np.exp(np.sum(dt[0] * A[None, :], axis=0))          # [H]
    assert np.max(np.abs(fi - (prod_a[None, :, None, None] * h0 + f0))) < 1e-12

    def seg_map(lo, hi):
        _, fz = oracle.ssd_scan(x[:, lo:hi], dt[:, lo:hi], A, B[:, lo:hi], C[:, lo:hi])
        return np.exp(np.sum(dt[0, lo:hi] * A[None, :], axis=0)), fz[0]

    (a1, b1), (a2, b2) = seg_map(0, 12), seg_map(12, 30)
    a12, b12 = a2 * a1, a2[:, None, None] * b1 + b2
    aw, bw = seg_map(0, 30)
    assert np.max(np.abs(a12 - aw)) < 1e-14 and np.max(np.abs(b12 - bw)) < 1e-12
    # non-commutative: swapping the order gives a different map
    b21 = a1[:, None, None] * b2 + b1
    assert np.max(np.abs(b21 - bw)) > 1e-3


def test_combine_operator_associative():
    rng = np.random.default_rng(12)
    comp = lambda s, f: (s[0] * f[0], s[0] * f[1] + s[1])   # s after f
    e = [(rng.uniform(0.1, 1), rng.standard_normal()) for _ in range(3)]
    l = comp(e[2], comp(e[1], e[0]))
    r = comp(comp(e[2], e[1]), e[0])
    assert abs(l[0] - r[0]) < 1e-15 and abs(l[1] - r[1]) < 1e-14


def test_varlen_equals_independent_runs():
    rng = np.random.default_rng(13)
    lens = [5, 0, 17, 1, 33]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    H, P, N, G = 4, 3, 5, 2
    x = rng.standard_normal((1, T, H, P))
    dt = rng.uniform(0.01, 0.4, (1, T, H))
    A = -rng.uniform(0.1, 2, H)
    B = rng.standard_normal((1, T, G, N))
    C = rng.standard_normal((1, T, G, N))
    D = rng.standard_normal(H)
    h0 = rng.standard_normal((len(lens), H, P, N))
    y, fin = oracle.ssd_scan(x, dt, A, B, C, D, h0, cu_seqlens=cu)
    for s in range(len(lens)):
        lo, hi = cu[s], cu[s + 1]
        ys, fs = oracle.ssd_scan(x[:, lo:hi], dt[:, lo:hi], A, B[:, lo:hi], C[:, lo:hi], D,
                                 h0[s:s + 1])
        assert np.max(np.abs(y[:, lo:hi] - ys), initial=0.0) < 1e-12
        assert np.max(np.abs(fin[s] - fs[0])) < 1e-12
    assert np.array_equal(fin[1], h0[1])   # empty sequence: final = init


def test_decode_steps_equal_scan():
    x, dt, A, B, C, D, h0 = _rand_problem(14, b=3, T=20)
    y, fin = oracle.ssd_scan(x, dt, A, B, C, D, h0)
    st = h0.copy()
    for t in range(x.shape[1]):
        yt, st = oracle.ssd_step(st, x[:, t], dt[:, t], A, B[:, t], C[:, t], D)
        assert np.max(np.abs(yt - y[:, t])) < 1e-12
    assert np.max(np.abs(st - fin)) < 1e-12


def test_group_mapping_contiguous():
    """Head h reads group floor(h*G/H): with G = H each head has its own B/C,
    and perturbing group g changes exactly heads g*H/G .. (g+1)*H/G - 1."""
    x, dt, A, B, C, D, _ = _rand_problem(15, b=1, T=12, H=6, G=3)
    y, _ = oracle.ssd_scan(x, dt, A, B, C, D)
    B2 = B.copy()
    B2[:, :, 1, :] += 1.0
    y2, _ = oracle.ssd_scan(x, dt, A, B2, C, D)
    changed = [h for h in range(6) if np.max(np.abs(y2[:, :, h] - y[:, :, h])) > 1e-9]
    assert changed == [2, 3]


def test_inputs_generator_recipe():
    """The generator's bf16 rounding is round-to-nearest-even and its value
    ranges follow the stated recipe."""
    bits, vals = I.bf16_round(np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-3],
                                       np.float32))
    assert list(vals[:3]) == [1.0, 1.0, 1.0 + 2 ** -6]   # ties go to even
    assert vals[3] == -2.5 and abs(vals[4] - 3.0e-3) < 3.0e-3 * 2 ** -8
    fi = I.make_forward_inputs(I.WORKLOADS["tiny_fp32"])
    assert fi.x.shape == (1, 256, 2, 16) and fi.init is None
    assert np.all(fi.A <= -1.0) and np.all(fi.A >= -16.0)
    assert np.all(fi.dt > 0)
    vl = I.make_forward_inputs(I.Workload("v", 1, 0, 2, 4, 4, 1, 64, "bf16", "zero", nseq=64,
                                          seed=1003))
    lens = np.diff(vl.cu_seqlens)
    assert len(lens) == 64 and lens.min() >= 64 and lens.max() < 8192
    assert vl.x.shape[1] == vl.cu_seqlens[-1]


def test_softplus_pins():
    # softplus(0) = ln 2; softplus(v) - softplus(-v) = v; softplus(v) -> v for
    # large v and -> exp(v) for very negative v
    import math
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    v = np.linspace(-30, 30, 121)
    assert np.allclose(oracle.softplus(v) - oracle.softplus(-v), v, rtol=0, atol=1e-12)
    assert oracle.softplus(50.0) == pytest.approx(50.0, rel=1e-15)
    assert oracle.softplus(-40.0) == pytest.approx(math.exp(-40.0), rel=1e-12)
    assert np.allclose(oracle.softplus(v), np.log1p(np.exp(v)), rtol=1e-13, atol=0)


def test_silu_gate_pins():
    # silu(0) = 0; silu(z) - silu(-z) = z; silu(z) -> z for large z, -> 0 for
    # very negative z; the gate scales y linearly
    z = np.linspace(-20, 20, 81)
    one = np.ones_like(z)
    assert oracle.silu_gate(1.0, 0.0) == 0.0
    assert np.allclose(oracle.silu_gate(one, z) - oracle.silu_gate(one, -z), z, rtol=0, atol=1e-12)
    assert oracle.silu_gate(1.0, 40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.silu_gate(1.0, -40.0)) < 1e-15
    assert np.allclose(oracle.silu_gate(3.0 * one, z), 3.0 * oracle.silu_gate(one, z), rtol=1e-15)
    # silu(z) = z * sigmoid(z), with sigmoid(z) = (1 + tanh(z / 2)) / 2 (valid where
    # the tanh form keeps its relative precision)
    zz = np.linspace(-8, 20, 57)
    assert np.allclose(oracle.silu_gate(np.ones_like(zz), zz), zz * 0.5 * (1 + np.tanh(zz / 2)),
                       rtol=1e-12, atol=0)


# ---- the tolerance metric itself ---------------------------------------------

def test_rel_err_hand_computed_values():
    """rel_err = max |got - ref| / RMS(ref), with values worked by hand: a
    wrong denominator (max |ref| instead of the RMS, a sum, a broadcast slip)
    or a missing absolute value changes these numbers."""
    # max diff 1 (at the last entry); RMS(ref) = sqrt((1 + 4 + 16) / 3) = sqrt(7)
    assert oracle.rel_err([1.0, 2.0, 3.0], [1.0, 2.0, 4.0]) == pytest.approx(1.0 / np.sqrt(7.0), rel=1e-15)
    # the diff is negative: |got - ref| must be taken; RMS(ref) = sqrt((9 + 16) / 2)
    assert oracle.rel_err([3.0, 2.5], [3.0, 4.0]) == pytest.approx(1.5 / np.sqrt(12.5), rel=1e-15)
    # max != RMS: ref = [0, 0, 0, 10] has RMS 5 and max 10
    assert oracle.rel_err([0.0, 0.0, 1.0, 10.0], [0.0, 0.0, 0.0, 10.0]) == pytest.approx(0.2, rel=1e-15)
    # 2-D inputs: the max and the RMS run over every element
    ref = np.array([[1.0, -1.0], [1.0, -1.0]])
    got = ref + np.array([[0.0, 0.0], [0.0, 0.5]])
    assert oracle.rel_err(got, ref) == pytest.approx(0.5, rel=1e-15)


def test_rel_err_edge_cases():
    assert oracle.rel_err(np.zeros(0), np.zeros(0)) == 0.0
    assert oracle.rel_err(np.zeros((3, 0)), np.zeros((3, 0))) == 0.0
    # a zero reference: the absolute difference is reported
    assert oracle.rel_err([0.25, 0.0], [0.0, 0.0]) == 0.25
    assert oracle.rel_err([1.0, 2.0], [1.0, 2.0]) == 0.0
