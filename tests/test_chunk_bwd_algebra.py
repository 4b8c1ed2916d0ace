"""The chunkwise backward algebra (tests/chunk_model.py: chunk_step_bwd and
chunked_backward) against the fp64 oracle's reverse-mode gradients, which
central differences of the forward oracle pin.

The model is the reverse of the WY/UT chunk step, built the way a
tensor-core backward would be.  Its gate gradients use prefix and suffix
scans and split pair products, so no gradient divides by a gate, and gates
that are exactly 0 or -1 are part of every case.  Agreement is to fp64
rounding.
"""
import numpy as np
import pytest

import chunk_model as cm
import oracle


def case(seed, T, n, dv, special=None):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, n))
    k = rng.standard_normal((T, n))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    al = rng.uniform(-1, 1, (T, n))
    al[rng.random((T, n)) < 0.1] = -1.0
    al[rng.random((T, n)) < 0.05] = 0.0
    be = rng.uniform(0, 2, T)
    if special == "alpha0":
        al[:] = 0.0
    elif special == "reflect":
        al[:] = -1.0
        be[:] = 2.0
    elif special == "beta0":
        be[:] = 0.0
    h0 = rng.standard_normal((n, dv))
    dhT = rng.standard_normal((n, dv))
    dO = rng.standard_normal((T, dv))
    return q, k, v, al, be, dO, h0, dhT


def compare(q, k, v, al, be, dO, h0, dhT, C):
    got = cm.chunked_backward(q, k, v, al, be, dO, h0=h0, dhT=dhT, C=C)
    X = lambda a: np.asarray(a, dtype=np.float64)[None, None]
    ref = oracle.bwd(X(q), X(k), X(v), X(al), X(be), X(dO), h0=X(h0), dhT=X(dhT))
    for name, g, r in zip(("dq", "dk", "dv", "dalpha", "dbeta", "dh0"), got, ref):
        r = np.asarray(r)[0, 0]
        scale = max(np.max(np.abs(r)), 1e-300)
        assert np.max(np.abs(g - r)) <= 1e-12 * scale, (name, np.max(np.abs(g - r)), scale)


@pytest.mark.parametrize("C,T", [(8, 1), (8, 8), (8, 29), (16, 37), (16, 64)])
def test_chunked_backward_matches_oracle(C, T):
    compare(*case(800 + T, T, 5, 4), C=C)


@pytest.mark.parametrize("special", ["alpha0", "reflect", "beta0"])
def test_chunked_backward_degenerate_gates(special):
    compare(*case(810, 21, 4, 3, special=special), C=8)


def test_chunked_backward_rectangular():
    compare(*case(820, 40, 3, 6), C=16)


@pytest.mark.parametrize("C", [4, 8, 16])
def test_tree_form_of_gram_gradients(C):
    """The split-tree form of the Gram gradients (per level: dense products of
    gated operands, then prefix and suffix scans for the gates) equals the
    explicit pair-product form."""
    rng = np.random.default_rng(830 + C)
    n = 4
    q, k = rng.standard_normal((C, n)), rng.standard_normal((C, n))
    al = rng.uniform(-1, 1, (C, n))
    al[rng.random((C, n)) < 0.15] = 0.0
    al[rng.random((C, n)) < 0.1] = -1.0
    dGk = rng.standard_normal((C, C)) * np.tril(np.ones((C, C)), -1)
    dGq = rng.standard_normal((C, C)) * np.tril(np.ones((C, C)))
    for a, b in zip(cm.gated_grams_bwd(q, k, al, dGk, dGq),
                    cm.gated_grams_bwd_direct(q, k, al, dGk, dGq)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
