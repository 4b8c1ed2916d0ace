"""Pins of the fp64 oracle to facts the pages and the mathematics fix.

Each test names its source.  Together they are chosen so that a plausible
mistake in the oracle (a dropped term, a sign, a transposed operand, the
readout taken before the update, a gate applied to columns instead of rows)
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def one_seq(q, k, v, alpha, beta, h0=None, scale=1.0):
    """Run the oracle on a single (sequence, head): inputs [T, n] etc."""
    q, k, v, alpha = (np.asarray(x, dtype=np.float64)[None, None] for x in (q, k, v, alpha))
    beta = np.asarray(beta, dtype=np.float64)[None, None]
    if h0 is not None:
        h0 = np.asarray(h0, dtype=np.float64)[None, None]
    o, hT = oracle.fwd(q, k, v, alpha, beta, h0, scale=scale)
    return o[0, 0], hT[0, 0]


def transition(alpha, beta, k):
    """The one-step transition matrix A, read off the oracle: h0 = I, v = 0."""
    n = len(alpha)
    z = np.zeros((1, n))
    _, H1 = one_seq(z, [k], z, [alpha], [beta], h0=np.eye(n))
    return H1


def unit(x):
    x = np.asarray(x, dtype=np.float64)
    return x / np.linalg.norm(x)


def rand_admissible(rng, n):
    """alpha in [-1,1]^n (with exact -1, 0, 1 sprinkled in), beta in [0,2], unit k."""
    a = rng.uniform(-1, 1, n)
    a[rng.random(n) < 0.15] = -1.0
    a[rng.random(n) < 0.05] = 0.0
    a[rng.random(n) < 0.05] = 1.0
    return a, rng.uniform(0, 2), unit(rng.standard_normal(n))


# --- the pages' worked example ------------------------------------------------

def _load_worked_case():
    s0, traces = None, {}
    with open(os.path.join(GOLDEN, "bounded_case_study_worked_case.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            if line.startswith("S0"):
                s0 = np.array([float(x) for x in line.split()[1:]]).reshape(2, 2)
                continue
            lhs, rhs = line.split("->")
            tag, step, beta, k1, k2, v1, v2 = lhs.split()
            traces.setdefault(tag, []).append(
                (int(step), float(beta), [float(k1), float(k2)], [float(v1), float(v2)],
                 np.array([float(x) for x in rhs.split()]).reshape(2, 2)))
    return s0, traces


def test_worked_case_decay_and_correction():
    """Bounded case study, worked case A (per-channel decay of row i by a_i)
    and B (exact correction to [4,4], then 4*0.2^2 = 0.160 retained; 3.240 on
    channel 1)."""
    s0, traces = _load_worked_case()
    a = [0.9, 0.2]
    for tag, steps in traces.items():
        T = len(steps)
        beta = [s[1] for s in steps]
        k = [s[2] for s in steps]
        v = [s[3] for s in steps]
        q = np.zeros((T, 2))
        for t in range(1, T + 1):
            # state after t steps: run the first t tokens
            _, hT = one_seq(q[:t], k[:t], v[:t], [a] * t, beta[:t], h0=s0)
            np.testing.assert_allclose(hT, steps[t - 1][4], rtol=0, atol=1e-12,
                                       err_msg=f"trace {tag} step {t}")


def test_worked_case_readout_is_of_updated_state():
    """The readout o_t = H_t^T q_t reads the UPDATED state ("Complex KDA"
    slides, frame "CKDA keeps the original gate--delta--readout structure").
    With q = e2 at the write step the output is exactly v = [4, 4]."""
    s0, _ = _load_worked_case()
    o, _ = one_seq([[0, 0], [0, 1]], [[0, 1], [0, 1]], [[0, 0], [4, 4]],
                   [[0.9, 0.2]] * 2, [0.0, 1.0], h0=s0)
    np.testing.assert_allclose(o[1], [4.0, 4.0], atol=1e-12)
    # and at the decay-only step it is row 2 of Diag(a) S0 = [1.0, 0.2]
    np.testing.assert_allclose(o[0], [0.0, 0.0], atol=1e-12)
    o, _ = one_seq([[0, 1]], [[0, 1]], [[0, 0]], [[0.9, 0.2]], [0.0], h0=s0)
    np.testing.assert_allclose(o[0], [1.0, 0.2], atol=1e-12)


def test_scale_multiplies_the_query():
    rng = np.random.default_rng(5)
    T, n = 9, 4
    args = (rng.standard_normal((T, n)), [unit(x) for x in rng.standard_normal((T, n))],
            rng.standard_normal((T, n)), rng.uniform(-1, 1, (T, n)), rng.uniform(0, 2, T))
    o1, h1 = one_seq(*args)
    o2, h2 = one_seq(*args, scale=0.375)
    np.testing.assert_allclose(o2, 0.375 * o1, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(h1, h2)


# --- closed forms ---------------------------------------------------------------

def test_two_reflections_make_rotation():
    """"Complex KDA" slides, "Two reflections make a rotation in one update":
    k = (1,1)/sqrt2, beta = 2, alpha = (-1, 1) gives R_{pi/2}."""
    with open(os.path.join(GOLDEN, "two_reflections_rotation.txt")) as f:
        rows = [l.split("#")[0].strip() for l in f if l.split("#")[0].strip()]
    for row in rows:
        lhs, rhs = row.split("->")
        a1, a2, beta, theta = (float(x) for x in lhs.split())
        want = np.array([float(x) for x in rhs.split()]).reshape(2, 2)
        A = transition([a1, a2], beta, [math.cos(theta), math.sin(theta)])
        np.testing.assert_allclose(A, want, atol=1e-15)


@pytest.mark.parametrize("seed", range(6))
def test_eq2_closed_form_and_discriminant(seed):
    """Paper Sec. 3, Eq. (2): A = (I - 2kk^T) Diag(alpha, 1), k = (cos t, sin t)
    = [[-a cos2t, -sin2t], [-a sin2t, cos2t]]; Delta = (1-a)^2 cos^2 2t + 4a;
    Delta < 0 gives a complex pair of modulus sqrt(-a)."""
    rng = np.random.default_rng(100 + seed)
    for _ in range(50):
        a = rng.uniform(-1, 1)
        th = rng.uniform(0, math.pi / 2)
        A = transition([a, 1.0], 2.0, [math.cos(th), math.sin(th)])
        c2, s2 = math.cos(2 * th), math.sin(2 * th)
        want = np.array([[-a * c2, -s2], [-a * s2, c2]])
        np.testing.assert_allclose(A, want, atol=1e-14)
        delta = (1 - a) ** 2 * c2 ** 2 + 4 * a
        lam = np.linalg.eigvals(A)
        if delta < -1e-9:
            assert np.all(np.abs(lam.imag) > 0)
            np.testing.assert_allclose(np.abs(lam), math.sqrt(-a), rtol=1e-9)
        elif delta > 1e-9:
            assert np.all(np.abs(lam.imag) < 1e-12)


def test_lemma24_one_layer_clock():
    """Paper App. D.2, Lemma 24: beta = 2, alpha = (1, -1), k = (-sin(phi/2),
    cos(phi/2)) is a rotation by phi; from c0 = e1 the state visits
    c_i = (cos(pi i/m), sin(pi i/m)) with phi = pi/m and returns after 2m steps."""
    for m in (1, 2, 3, 5, 8):
        phi = math.pi / m
        T = 2 * m
        k = [[-math.sin(phi / 2), math.cos(phi / 2)]] * T
        qs = np.eye(2)[np.arange(T) % 2]  # any queries
        o, hT = one_seq(qs, k, np.zeros((T, 1)), [[1.0, -1.0]] * T, [2.0] * T,
                        h0=np.array([[1.0], [0.0]]))
        for i in range(1, T + 1):
            _, Hi = one_seq(qs[:i], k[:i], np.zeros((i, 1)), [[1.0, -1.0]] * i, [2.0] * i,
                            h0=np.array([[1.0], [0.0]]))
            np.testing.assert_allclose(Hi[:, 0], [math.cos(math.pi * i / m),
                                                  math.sin(math.pi * i / m)], atol=1e-13)
            np.testing.assert_allclose(o[i - 1, 0], qs[i - 1] @ Hi[:, 0], atol=1e-13)
        np.testing.assert_allclose(hT[:, 0], [1.0, 0.0], atol=1e-13)


@pytest.mark.parametrize("seed", range(4))
def test_prop2_sign_core_block(seed):
    """Paper Prop. 2 / App. A.2 (Prop. 7), slides backup "separate the sign core
    from magnitude scaling": with unit gates of mixed sign, (I - beta kk^T) S
    restricted to span(k-, k+) is [[b c^2 - 1, -b s c], [b s c, 1 - b s^2]] in
    the basis (k-/|k-|, k+/|k+|), |k-| = cos th, |k+| = sin th; the complement
    keeps its signs."""
    rng = np.random.default_rng(200 + seed)
    n = 6
    sgn = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    sgn[0], sgn[1] = -1.0, 1.0
    th = rng.uniform(0.1, 1.4)
    beta = rng.uniform(0, 2)
    um = np.where(sgn < 0, rng.standard_normal(n), 0.0)
    up = np.where(sgn > 0, rng.standard_normal(n), 0.0)
    um, up = unit(um), unit(up)
    k = math.cos(th) * um + math.sin(th) * up
    A = transition(sgn, beta, k)
    c, s = math.cos(th), math.sin(th)
    basis = np.stack([um, up], axis=1)
    blk = basis.T @ A @ basis
    np.testing.assert_allclose(blk, [[beta * c * c - 1, -beta * s * c],
                                     [beta * s * c, 1 - beta * s * s]], atol=1e-13)
    # A maps the plane to itself
    np.testing.assert_allclose(A @ basis, basis @ blk, atol=1e-13)
    # on the orthogonal complement A acts as the sign diagonal
    P = np.eye(n) - basis @ basis.T
    np.testing.assert_allclose(A @ P, np.diag(sgn) @ P, atol=1e-13)
    if abs(beta - 2.0) < 1e-15:
        pass
    # at beta = 2 the block is the rotation by 2 theta
    A2 = transition(sgn, 2.0, k)
    blk2 = basis.T @ A2 @ basis
    np.testing.assert_allclose(blk2, [[math.cos(2 * th), -math.sin(2 * th)],
                                      [math.sin(2 * th), math.cos(2 * th)]], atol=1e-13)


def test_eq3_diagonal_as_axis_householders():
    """Paper Sec. 3, Eq. (3): Diag(alpha) = prod_i (I - (1 - alpha_i) e_i e_i^T).
    With beta = 1 - alpha_i and k = e_i, the oracle's transition with a unit
    gate is exactly that axis factor; chaining n such steps gives Diag(alpha)."""
    rng = np.random.default_rng(7)
    n = 5
    alpha = rng.uniform(-1, 1, n)
    T = n
    k = np.eye(n)
    _, H = one_seq(np.zeros((T, n)), k, np.zeros((T, n)), np.ones((T, n)), 1.0 - alpha,
                   h0=np.eye(n))
    np.testing.assert_allclose(H, np.diag(alpha), atol=1e-15)


# --- invariants -------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_non_expansive_transition(seed):
    """Slides, "The transition remains non-expansive and inexpensive":
    ||A_t||_2 <= ||I - beta kk^T||_2 ||Diag alpha||_2 <= 1; with v = 0 the state
    norm never grows; additive writes can grow it."""
    rng = np.random.default_rng(300 + seed)
    n = 8
    for _ in range(40):
        a, b, k = rand_admissible(rng, n)
        A = transition(a, b, k)
        assert np.linalg.norm(A, 2) <= 1.0 + 1e-12
    T = 30
    ks = [unit(x) for x in rng.standard_normal((T, n))]
    al = rng.uniform(-1, 1, (T, n))
    be = rng.uniform(0, 2, T)
    h0 = rng.standard_normal((n, 3))
    prev = np.linalg.norm(h0, 2)
    for t in range(1, T + 1):
        _, Ht = one_seq(np.zeros((t, n)), ks[:t], np.zeros((t, 3)), al[:t], be[:t], h0=h0)
        cur = np.linalg.norm(Ht, 2)
        assert cur <= prev * (1 + 1e-12) + 1e-14
        prev = cur
    # a write can increase the norm
    _, Hw = one_seq(np.zeros((1, n)), [np.eye(n)[0]], [[5.0, 0, 0]], [np.ones(n)], [1.0],
                    h0=np.zeros((n, 3)))
    assert np.linalg.norm(Hw, 2) > 4.9


@pytest.mark.parametrize("seed", range(4))
def test_spectrum_theorem8(seed):
    """Paper App. A.3, Thm. 8 (slides table "Both range extensions are needed"):
    a CKDA transition has at most one non-real conjugate pair; none when
    beta <= 1 or when every alpha >= 0."""
    rng = np.random.default_rng(400 + seed)
    n = 6
    for _ in range(60):
        a, b, k = rand_admissible(rng, n)
        lam = np.linalg.eigvals(transition(a, b, k))
        assert np.sum(np.abs(lam.imag) > 1e-9) <= 2
        lam1 = np.linalg.eigvals(transition(a, rng.uniform(0, 1), k))
        assert np.all(np.abs(lam1.imag) < 1e-9)
        lam2 = np.linalg.eigvals(transition(np.abs(a), b, k))
        assert np.all(np.abs(lam2.imag) < 1e-9)
    # and the pair does occur for the rotation example
    lam = np.linalg.eigvals(transition([-1.0, 1.0], 2.0, unit([1, 1])))
    assert np.sum(np.abs(lam.imag) > 0.5) == 2


@pytest.mark.parametrize("seed", range(3))
def test_signed_householder_products_are_orthogonal(seed):
    """Paper Thm. 1 / App. B.3 (signed-Householder family SH_d): with
    alpha in {-1, 1}^n and beta in {0, 2} every transition is orthogonal, so
    from h0 = I with v = 0 the final state is orthogonal."""
    rng = np.random.default_rng(500 + seed)
    n, T = 7, 40
    al = np.where(rng.random((T, n)) < 0.5, -1.0, 1.0)
    be = np.where(rng.random(T) < 0.7, 2.0, 0.0)
    ks = [unit(x) for x in rng.standard_normal((T, n))]
    _, H = one_seq(np.zeros((T, n)), ks, np.zeros((T, n)), al, be, h0=np.eye(n))
    np.testing.assert_allclose(H.T @ H, np.eye(n), atol=1e-12)


# --- brute force ---------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(8))
def test_brute_force_dense_transitions(seed):
    """Paper Eq. (1) / App. B.2 Eq. (9) with the transition materialised as an
    explicit n x n matrix, A_t = (I - beta_t k_t k_t^T) Diag(alpha_t), and
    H_t = A_t H_{t-1} + beta_t k_t v_t^T, o_t = H_t^T q_t."""
    rng = np.random.default_rng(600 + seed)
    n = int(rng.integers(1, 9))
    dv = int(rng.integers(1, 9))
    T = int(rng.integers(1, 65))
    q = rng.standard_normal((T, n))
    k = np.stack([unit(x) for x in rng.standard_normal((T, n))])
    v = rng.standard_normal((T, dv))
    al = rng.uniform(-1, 1, (T, n))
    al[rng.random((T, n)) < 0.1] = -1.0
    al[rng.random((T, n)) < 0.05] = 0.0
    be = rng.uniform(0, 2, T)
    h0 = rng.standard_normal((n, dv)) if seed % 2 else np.zeros((n, dv))
    o, hT = one_seq(q, k, v, al, be, h0=h0)
    H = h0.copy()
    for t in range(T):
        A = (np.eye(n) - be[t] * np.outer(k[t], k[t])) @ np.diag(al[t])
        H = A @ H + be[t] * np.outer(k[t], v[t])
        np.testing.assert_allclose(o[t], H.T @ q[t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hT, H, rtol=1e-12, atol=1e-12)


def test_homogeneous_product_is_product_of_transitions():
    """With v = 0 and h0 = I the final state is the ordered product A_T ... A_1."""
    rng = np.random.default_rng(11)
    n, T = 5, 20
    k = np.stack([unit(x) for x in rng.standard_normal((T, n))])
    al = rng.uniform(-1, 1, (T, n))
    be = rng.uniform(0, 2, T)
    _, H = one_seq(np.zeros((T, n)), k, np.zeros((T, n)), al, be, h0=np.eye(n))
    P = np.eye(n)
    for t in range(T):
        P = (np.eye(n) - be[t] * np.outer(k[t], k[t])) @ np.diag(al[t]) @ P
    np.testing.assert_allclose(H, P, atol=1e-13)


# --- equivalences --------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(3))
def test_sign_gauge_equivalence(seed):
    """Slides, "Absorb cumulative signs into keys and queries" (paper Lemma 27):
    with S_t = Diag(sign alpha_t) (sign(0) = +1, paper App. A.2), P_t = S_1..S_t,
    running on (P_t k_t, P_t q_t, |alpha_t|) gives the same outputs, and the
    final state is P_T H_T."""
    rng = np.random.default_rng(700 + seed)
    n, dv, T = 6, 4, 50
    q = rng.standard_normal((T, n))
    k = np.stack([unit(x) for x in rng.standard_normal((T, n))])
    v = rng.standard_normal((T, dv))
    al = rng.uniform(-1, 1, (T, n))
    al[rng.random((T, n)) < 0.1] = 0.0
    al[rng.random((T, n)) < 0.1] = -1.0
    be = rng.uniform(0, 2, T)
    h0 = rng.standard_normal((n, dv))
    o, hT = one_seq(q, k, v, al, be, h0=h0)
    s = np.where(al < 0, -1.0, 1.0)
    P = np.cumprod(s, axis=0)
    o2, hT2 = one_seq(P * q, P * k, v, np.abs(al), be, h0=h0)
    np.testing.assert_allclose(o2, o, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(hT2, P[-1][:, None] * hT, rtol=1e-11, atol=1e-11)


def test_channel_permutation_equivariance():
    """Adapted from "On State Reduction in Linear Attention", Prop. 3.1 (an
    orthogonal change of key/query basis leaves the output unchanged): a
    permutation commutes with Diag(alpha), so permuting the channels of q, k,
    alpha and the rows of h0 leaves o unchanged and permutes the rows of hT."""
    rng = np.random.default_rng(12)
    n, dv, T = 7, 3, 33
    q = rng.standard_normal((T, n))
    k = np.stack([unit(x) for x in rng.standard_normal((T, n))])
    v = rng.standard_normal((T, dv))
    al = rng.uniform(-1, 1, (T, n))
    be = rng.uniform(0, 2, T)
    h0 = rng.standard_normal((n, dv))
    perm = rng.permutation(n)
    o, hT = one_seq(q, k, v, al, be, h0=h0)
    o2, hT2 = one_seq(q[:, perm], k[:, perm], v, al[:, perm], be, h0=h0[perm])
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hT2, hT[perm], rtol=1e-12, atol=1e-12)


def test_reductions():
    """alpha = 1, beta = 0: the state never changes and o_t = h0^T q_t.
    beta = 1 on a unit key: exact correction, H_t^T k_t = v_t (bounded case
    study, "Delta correction": the write lands exactly)."""
    rng = np.random.default_rng(13)
    n, dv, T = 6, 5, 17
    q = rng.standard_normal((T, n))
    k = np.stack([unit(x) for x in rng.standard_normal((T, n))])
    v = rng.standard_normal((T, dv))
    h0 = rng.standard_normal((n, dv))
    o, hT = one_seq(q, k, v, np.ones((T, n)), np.zeros(T), h0=h0)
    np.testing.assert_allclose(o, q @ h0, atol=1e-13)
    np.testing.assert_allclose(hT, h0, atol=0)
    al = rng.uniform(-1, 1, (T, n))
    o, _ = one_seq(k, k, v, al, np.ones(T), h0=h0)
    np.testing.assert_allclose(o, v, atol=1e-12)
    # alpha = 0 on every channel erases the past: the state is the fresh write
    o, hT = one_seq(q[:1], k[:1], v[:1], np.zeros((1, n)), [0.7], h0=h0)
    np.testing.assert_allclose(hT, 0.7 * np.outer(k[0], v[0]), atol=1e-14)


# --- batching, packing and resume (host logic of the oracle) ----------------------

def test_packed_equals_separate_and_resume_split():
    rng = np.random.default_rng(14)
    H, n, dv = 3, 4, 5
    lengths = [5, 1, 0, 9, 3]
    Tt = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q = rng.standard_normal((1, H, Tt, n))
    k = rng.standard_normal((1, H, Tt, n))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, H, Tt, dv))
    al = rng.uniform(-1, 1, (1, H, Tt, n))
    be = rng.uniform(0, 2, (1, H, Tt))
    h0 = rng.standard_normal((len(lengths), H, n, dv))
    o, hT = oracle.fwd(q, k, v, al, be, h0, cu_seqlens=cu)
    for s, L in enumerate(lengths):
        a, b = cu[s], cu[s + 1]
        o1, h1 = oracle.fwd(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], al[:, :, a:b],
                            be[:, :, a:b], h0[s:s + 1])
        np.testing.assert_array_equal(o[:, :, a:b], o1)
        np.testing.assert_array_equal(hT[s:s + 1], h1)
    # resume: fwd(T) == fwd(T1) then fwd(T2, h0 = hT1)
    sl = slice(0, 9)
    x = [t[:, :, cu[3]:cu[4]] for t in (q, k, v, al, be)]
    oa, ha = oracle.fwd(*x, h0[3:4])
    x1 = [t[:, :, :4] for t in x]
    x2 = [t[:, :, 4:] for t in x]
    o1, h1 = oracle.fwd(*x1, h0[3:4])
    o2, h2 = oracle.fwd(*x2, h1)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=2), oa, rtol=0, atol=1e-15)
    np.testing.assert_allclose(h2, ha, rtol=0, atol=1e-15)
    del sl


@pytest.mark.parametrize("dk,dv", [(6, 6), (4, 7)])
def test_segment_operators_compose(dk, dv):
    """Paper Eq. (1) read over a run of tokens: the final state is affine in
    the initial one, H_out = P H_in + F, with P the product of the run's
    transitions (the final state from [I | 0] with v = 0) and F the final
    state from zero.  Chaining segment operators by that scan, and then
    rerunning each segment from its scanned state, gives the outputs and final
    state of one pass (the bounded case study's "Chunkwise execution": an
    execution strategy that changes cost, never the numbers)."""
    rng = np.random.default_rng(700 + dk)
    T, cuts = 37, [0, 12, 24, 37]
    q = rng.standard_normal((1, 1, T, dk))
    k = rng.standard_normal((1, 1, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, 1, T, dv))
    al = rng.uniform(-1, 1, (1, 1, T, dk))
    al[rng.random(al.shape) < 0.1] = -1.0
    al[rng.random(al.shape) < 0.05] = 0.0
    be = rng.uniform(0, 2, (1, 1, T))
    h0 = rng.standard_normal((1, 1, dk, dv))
    o_ref, h_ref = oracle.fwd(q, k, v, al, be, h0)
    seg = lambda x, s: x[:, :, cuts[s]:cuts[s + 1]]
    eye = np.zeros((1, 1, dk, dv))
    eye[0, 0, :, :min(dk, dv)] = np.eye(dk, min(dk, dv))
    # the affine map of one segment, checked on a random initial state
    x1 = [seg(t, 1) for t in (q, k, v, al, be)]
    _, F1 = oracle.fwd(*x1, None)
    if dk <= dv:
        _, PI = oracle.fwd(x1[0], x1[1], np.zeros_like(x1[2]), x1[3], x1[4], eye)
        P1 = PI[0, 0, :, :dk]
        assert np.all(PI[0, 0, :, dk:] == 0.0)
        _, Hr = oracle.fwd(*x1, h0)
        np.testing.assert_allclose(Hr[0, 0], P1 @ h0[0, 0] + F1[0, 0], rtol=0, atol=1e-12)
    # the split's two passes and scan, with the oracle for every pass
    outs, H = [], None
    for s_ in range(len(cuts) - 1):
        xs = [seg(t, s_) for t in (q, k, v, al, be)]
        if s_ == 0:
            o_s, H = oracle.fwd(*xs, h0)
        else:
            o_s, H_next = oracle.fwd(*xs, H)
            # the state after the segment from the scan: P H + F
            _, Fs = oracle.fwd(*xs, None)
            Hz = np.zeros((1, 1, dk, dv))
            for c in range(dv):   # P applied column by column: v = 0, h0 = e_c in column c
                e_c = np.zeros((1, 1, dk, dv))
                e_c[0, 0, :, c] = H[0, 0, :, c]
                _, Pc = oracle.fwd(xs[0], xs[1], np.zeros_like(xs[2]), xs[3], xs[4], e_c)
                Hz[0, 0, :, c] = Pc[0, 0, :, c]
            np.testing.assert_allclose(H_next, Hz + Fs, rtol=0, atol=1e-12)
            H = H_next
        outs.append(o_s)
    np.testing.assert_allclose(np.concatenate(outs, axis=2), o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(H, h_ref, rtol=0, atol=1e-12)


def test_decode_step_matches_fwd_token_by_token():
    rng = np.random.default_rng(15)
    B, H, n, dv, T = 2, 3, 5, 4, 6
    q = rng.standard_normal((B, H, T, n))
    k = rng.standard_normal((B, H, T, n))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    al = rng.uniform(-1, 1, (B, H, T, n))
    be = rng.uniform(0, 2, (B, H, T))
    h0 = rng.standard_normal((B, H, n, dv))
    o, hT = oracle.fwd(q, k, v, al, be, h0, scale=0.5)
    S = h0.copy()
    for t in range(T):
        ot, S = oracle.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], al[:, :, t],
                                   be[:, :, t], S, scale=0.5)
        np.testing.assert_array_equal(ot, o[:, :, t])
    np.testing.assert_array_equal(S, hT)


def test_oracle_rejects_bad_packing():
    z = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        oracle.fwd(z, z, z, z, np.zeros((1, 1, 4)), cu_seqlens=[0, 3])
    with pytest.raises(ValueError):
        oracle.fwd(z, z, z, z, np.zeros((1, 1, 4)), cu_seqlens=[0, 3, 2, 4])


# ----------------------------------------------------------------- input prep
# "Complex KDA" discussion slides, backup frame "practical gates differ from
# exact theoretical endpoints": r = tanh(a/2), alpha = s[eps + (1-eps)|r|]
# with eps = e^-5 and s = +1 for r >= 0, -1 otherwise; beta = 2 sigma(b);
# log|alpha| stays in [-5, 0]; finite logits approach but do not attain
# |alpha| = 1 or beta = 2.  Keys have unit norm (paper Sec. 2).

def _prep_gates(a, b):
    a = np.asarray(a, dtype=np.float64).reshape(1, -1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)[:1]
    k = np.ones_like(a)
    _, _, alpha, beta = oracle.prep(k, a, b)
    return alpha[0], beta


def test_prep_sign_rule_and_zero():
    """s = +1 for r >= 0 (so a = 0 and a = -0 give +e^-5), -1 for r < 0."""
    a = np.array([0.0, -0.0, 1e-30, -1e-30, 0.3, -0.3, 7.0, -7.0])
    alpha, _ = _prep_gates(a, [0.0])
    assert alpha[0] == math.exp(-5.0) and alpha[1] == math.exp(-5.0)
    np.testing.assert_array_equal(np.sign(alpha[2:]), [1, -1, 1, -1, 1, -1])
    # next to a = 0 the gate jumps between the two endpoints +-e^-5
    assert alpha[2] == pytest.approx(math.exp(-5.0), rel=1e-12)
    assert alpha[3] == pytest.approx(-math.exp(-5.0), rel=1e-12)


def test_prep_gate_range_and_endpoints():
    """log|alpha| in [-5, 0] for every logit; |alpha| and beta approach 1 and
    2 (or 0) for large logits; beta(0) = 1 (sigma(0) = 1/2)."""
    a = np.linspace(-60.0, 60.0, 2001)
    alpha, _ = _prep_gates(a, [0.0])
    la = np.log(np.abs(alpha))
    assert la.min() >= -5.0 - 1e-12 and la.max() <= 0.0
    assert abs(alpha[-1]) == pytest.approx(1.0, abs=1e-12)
    assert abs(alpha[0]) == pytest.approx(1.0, abs=1e-12)
    # finite moderate logits stay strictly inside
    alpha_mid, _ = _prep_gates([8.0, -8.0], [0.0])
    assert np.all(np.abs(alpha_mid) < 1.0)
    for b, want in ((0.0, 1.0), (40.0, 2.0), (-40.0, 0.0)):
        _, beta = _prep_gates([0.0], [b])
        assert beta[0] == pytest.approx(want, abs=1e-12)
    _, beta = _prep_gates([0.0], [5.0])
    assert 0.0 < beta[0] < 2.0


def test_prep_symmetries_and_monotonicity():
    """alpha(-a) = -alpha(a) for a != 0 (tanh is odd, s flips); beta(-b) =
    2 - beta(b) (sigma(-b) = 1 - sigma(b)); |alpha| grows with |a|."""
    rng = np.random.default_rng(5)
    a = rng.normal(0.0, 3.0, 257)
    a = a[a != 0.0]
    ap, _ = _prep_gates(a, [0.0])
    am, _ = _prep_gates(-a, [0.0])
    np.testing.assert_allclose(am, -ap, rtol=0, atol=1e-15)
    for b in rng.normal(0.0, 4.0, 16):
        _, bp = _prep_gates([0.0], [b])
        _, bm = _prep_gates([0.0], [-b])
        assert bp[0] + bm[0] == pytest.approx(2.0, abs=1e-14)
    grid = np.linspace(0.0, 30.0, 301)
    g, _ = _prep_gates(grid, [0.0])
    assert np.all(np.diff(g) >= 0.0)


def test_prep_half_logit_scale():
    """r = tanh(a/2): a gate with a = 2 atanh(r*) has |r| = r*, so alpha =
    eps + (1 - eps) r* -- e.g. r* = 1/2 at a = ln 3 (tanh(ln(3)/2) = 1/2)."""
    alpha, _ = _prep_gates([math.log(3.0)], [0.0])
    eps = math.exp(-5.0)
    assert alpha[0] == pytest.approx(eps + (1.0 - eps) * 0.5, rel=1e-14)


def test_prep_unit_keys():
    """Normalised keys have unit norm and point along the raw key; q is
    normalised only on request (else copied); zero keys stay finite."""
    rng = np.random.default_rng(6)
    k = rng.normal(0.0, 1.0, (9, 24)) * rng.uniform(0.1, 10.0, (9, 1))
    q = rng.normal(0.0, 1.0, (9, 24))
    a = np.zeros_like(k)
    b = np.zeros(9)
    qn, kn, _, _ = oracle.prep(k, a, b, q_raw=q, normalize_q=True, norm_eps=0.0)
    np.testing.assert_allclose(np.linalg.norm(kn, axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(qn, axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(np.sum(kn * k, axis=1), np.linalg.norm(k, axis=1), rtol=1e-13)
    qc, _, _, _ = oracle.prep(k, a, b, q_raw=q, normalize_q=False)
    np.testing.assert_array_equal(qc, q)
    _, kz, _, _ = oracle.prep(np.zeros((1, 8)), np.zeros((1, 8)), np.zeros(1))
    assert np.all(kz == 0.0)


# ------------------------------------------------------------------ backward
# The backward is pinned to the forward oracle (itself pinned above) by
# central finite differences of L = sum_t <o_t, do_t> + <hT, dhT>: a wrong
# sign, a dropped term or a transposed operand anywhere in the reverse steps
# moves some gradient by O(1) relative, far outside the O(h^2) difference
# error.

def _loss(x, do, dhT, scale):
    o, hT = oracle.fwd(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["h0"],
                       cu_seqlens=x.get("cu"), scale=scale)
    return float(np.sum(o * do) + np.sum(hT * dhT))


def _fd_case(seed, B=1, H=2, T=7, dk=3, dv=2, special=False, cu=None):
    rng = np.random.default_rng(seed)
    x = {"q": rng.normal(size=(B, H, T, dk)), "k": rng.normal(size=(B, H, T, dk)),
         "v": rng.normal(size=(B, H, T, dv)), "alpha": rng.uniform(-1, 1, (B, H, T, dk)),
         "beta": rng.uniform(0, 2, (B, H, T)), "h0": None}
    x["k"] /= np.linalg.norm(x["k"], axis=-1, keepdims=True)
    N = B if cu is None else len(cu) - 1
    x["h0"] = rng.normal(size=(N, H, dk, dv))
    if cu is not None:
        x["cu"] = np.asarray(cu, dtype=np.int32)
    if special:
        x["alpha"][..., 1, 0] = 0.0
        x["alpha"][..., 3, :] = -1.0
        x["beta"][..., 2] = 2.0
        x["beta"][..., 4] = 0.0
    do = rng.normal(size=(B, H, T, dv))
    dhT = rng.normal(size=(N, H, dk, dv))
    return x, do, dhT


@pytest.mark.parametrize("special", [False, True])
def test_bwd_matches_central_differences(special):
    scale = 0.8
    x, do, dhT = _fd_case(3 + special, special=special)
    g = oracle.bwd(x["q"], x["k"], x["v"], x["alpha"], x["beta"], do, h0=x["h0"], dhT=dhT,
                   scale=scale)
    names = ["q", "k", "v", "alpha", "beta", "h0"]
    h = 1e-6
    for name, grad in zip(names, g):
        base = x[name]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = base[idx]
            base[idx] = old + h
            lp = _loss(x, do, dhT, scale)
            base[idx] = old - h
            lm = _loss(x, do, dhT, scale)
            base[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - grad)) / max(np.max(np.abs(num)), 1e-12)
        assert err < 1e-7, (name, err)


def test_bwd_packed_matches_central_differences():
    cu = [0, 3, 3, 7]
    x, do, dhT = _fd_case(11, B=1, H=2, T=7, cu=cu)
    g = oracle.bwd(x["q"], x["k"], x["v"], x["alpha"], x["beta"], do, h0=x["h0"], dhT=dhT,
                   cu_seqlens=x["cu"])
    h = 1e-6
    for name, grad in zip(["k", "alpha", "h0"], (g[1], g[3], g[5])):
        base = x[name]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = base[idx]
            base[idx] = old + h
            lp = _loss(x, do, dhT, 1.0)
            base[idx] = old - h
            lm = _loss(x, do, dhT, 1.0)
            base[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - grad)) / max(np.max(np.abs(num)), 1e-12)
        assert err < 1e-7, (name, err)


def test_bwd_closed_form_without_writes_or_decay():
    """beta = 0 and alpha = 1: H_t = h0 for every t, o_t = h0^T (s q_t).  Then
    dq_t = s h0 do_t, dh0 = s sum_t q_t do_t^T + dhT, dv = 0, dalpha_t,i =
    sum_j D_t,ij (h0)_ij with D_t = dhT + s sum_{r >= t} q_r do_r^T."""
    rng = np.random.default_rng(21)
    T, n, dv, s = 5, 4, 3, 1.5
    q = rng.normal(size=(1, 1, T, n))
    k = rng.normal(size=(1, 1, T, n))
    v = rng.normal(size=(1, 1, T, dv))
    a = np.ones((1, 1, T, n))
    b = np.zeros((1, 1, T))
    h0 = rng.normal(size=(1, 1, n, dv))
    do = rng.normal(size=(1, 1, T, dv))
    dhT = rng.normal(size=(1, 1, n, dv))
    dq, _, dvv, dal, _, dh0 = oracle.bwd(q, k, v, a, b, do, h0=h0, dhT=dhT, scale=s)
    H0 = h0[0, 0]
    for t in range(T):
        np.testing.assert_allclose(dq[0, 0, t], s * H0 @ do[0, 0, t], rtol=1e-13)
        D = dhT[0, 0] + s * sum(np.outer(q[0, 0, r], do[0, 0, r]) for r in range(t, T))
        np.testing.assert_allclose(dal[0, 0, t], np.sum(D * H0, axis=1), rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(dvv, 0.0)
    want = dhT[0, 0] + s * sum(np.outer(q[0, 0, t], do[0, 0, t]) for t in range(T))
    np.testing.assert_allclose(dh0[0, 0], want, rtol=1e-12)


# ------------------------------------------------------- input prep backward
# The gradients of prep's outputs with respect to its raw inputs.  Pinned by
# central differences of prep itself (pinned above), away from a = 0 where
# the gate's sign jumps; at a = 0 by the reading that the sign carries no
# gradient and |tanh(a/2)| takes the subgradient 0.

def _prep_loss(w, q_raw, k_raw, a_raw, b_raw, normalize_q, norm_eps):
    """L = <wq, q> + <wk, k> + <wa, alpha> + <wb, beta> of prep's outputs."""
    q, k, alpha, beta = oracle.prep(k_raw, a_raw, b_raw, q_raw=q_raw,
                                    normalize_q=normalize_q, norm_eps=norm_eps)
    wq, wk, wa, wb = w
    return float(np.sum(wq * q) + np.sum(wk * k) + np.sum(wa * alpha) + np.sum(wb * beta))


@pytest.mark.parametrize("normalize_q,norm_eps", [(True, 1e-6), (True, 0.0), (False, 1e-3)])
def test_prep_bwd_central_differences(normalize_q, norm_eps):
    rng = np.random.default_rng(60)
    R, n = 4, 6
    q_raw = rng.normal(0.0, 1.0, (R, n)) * rng.uniform(0.2, 5.0, (R, 1))
    k_raw = rng.normal(0.0, 1.0, (R, n)) * rng.uniform(0.2, 5.0, (R, 1))
    a_raw = rng.normal(0.0, 2.0, (R, n))
    a_raw = np.where(np.abs(a_raw) < 0.05, 0.3, a_raw)     # the sign is constant nearby
    b_raw = rng.normal(0.0, 2.0, R)
    w = (rng.normal(size=(R, n)), rng.normal(size=(R, n)), rng.normal(size=(R, n)),
         rng.normal(size=R))
    dq_raw, dk_raw, da_raw, db_raw = oracle.prep_bwd(
        k_raw, a_raw, b_raw, w[1], w[2], w[3], q_raw=q_raw, dq=w[0],
        normalize_q=normalize_q, norm_eps=norm_eps)
    args = [q_raw, k_raw, a_raw, b_raw]
    for which, got in enumerate((dq_raw, dk_raw, da_raw, db_raw)):
        x = args[which]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            h = 1e-6 * max(1.0, abs(x[idx]))
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            ap, am = list(args), list(args)
            ap[which], am[which] = xp, xm
            num[idx] = (_prep_loss(w, *ap, normalize_q, norm_eps)
                        - _prep_loss(w, *am, normalize_q, norm_eps)) / (2 * h)
        np.testing.assert_allclose(got, num, rtol=1e-6, atol=1e-8, err_msg=str(which))


def test_prep_bwd_gate_at_zero_and_closed_forms():
    """At a = 0 the gate gradient is 0 (sign detached, subgradient 0 of |r|);
    next to 0 it is (1 - e^-5)/2 from either side, as the one-sided
    differences give; dbeta/db = 1/2 at b = 0 and vanishes without NaN for
    huge |b|."""
    eps = math.exp(-5.0)
    a = np.array([[0.0, -0.0, 1e-4, -1e-4]])
    k = np.ones_like(a)
    ones = np.ones_like(a)
    _, _, da, db = oracle.prep_bwd(k, a, np.array([0.0]), np.zeros_like(a), ones,
                                   np.array([1.0]))
    assert da[0, 0] == 0.0 and da[0, 1] == 0.0
    assert db[0] == 0.5
    # one-sided differences on each side of 0 (where s is constant)
    for x0, g in ((1e-4, da[0, 2]), (-1e-4, da[0, 3])):
        h = 1e-7
        _, _, ap, _ = oracle.prep(np.ones((1, 1)), np.array([[x0 + h]]), np.zeros(1))
        _, _, am, _ = oracle.prep(np.ones((1, 1)), np.array([[x0 - h]]), np.zeros(1))
        assert g == pytest.approx((ap[0, 0] - am[0, 0]) / (2 * h), rel=1e-7)
        assert g == pytest.approx((1.0 - eps) / 2.0, rel=1e-7)
    _, _, _, db = oracle.prep_bwd(np.ones((2, 1)), np.ones((2, 1)), np.array([800.0, -800.0]),
                                  np.zeros((2, 1)), np.zeros((2, 1)), np.ones(2))
    assert np.all(np.isfinite(db)) and np.all(np.abs(db) < 1e-300)


def test_prep_bwd_invariances():
    """k / |k| is scale-invariant, so with norm_eps = 0 the key gradient is
    orthogonal to the raw key; an unnormalised q passes its gradient through."""
    rng = np.random.default_rng(61)
    k = rng.normal(size=(7, 16)) * 3.0
    q = rng.normal(size=(7, 16))
    dk = rng.normal(size=(7, 16))
    dq = rng.normal(size=(7, 16))
    z = np.zeros((7, 16))
    dq_raw, dk_raw, _, _ = oracle.prep_bwd(k, z, np.zeros(7), dk, z, np.zeros(7), q_raw=q, dq=dq,
                                           normalize_q=False, norm_eps=0.0)
    np.testing.assert_allclose(np.sum(dk_raw * k, axis=1), 0.0, atol=1e-13)
    np.testing.assert_array_equal(dq_raw, dq)
