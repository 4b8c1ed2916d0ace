"""The division-free chunk decomposition reaches the token recurrence exactly.

Checks the algebra the CUDA forward kernel is built on (tests/chunk_model.py)
against the fp64 oracle, in fp64, on gates that include exact zeros and -1,
ragged tails, and every chunk size the kernels use.
"""
import numpy as np
import pytest

import oracle
from chunk_model import chunked_forward, gated_grams


def _inputs(rng, T, n, dv, zeros=0.05, negs=0.1):
    q = rng.standard_normal((T, n))
    k = rng.standard_normal((T, n))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    a = np.tanh(2 * rng.standard_normal((T, n)))
    u = rng.random((T, n))
    a[u < zeros] = 0.0
    a[(u >= zeros) & (u < zeros + negs)] = -1.0
    b = 2 / (1 + np.exp(-rng.standard_normal(T)))
    return q, k, v, a, b


@pytest.mark.parametrize("C", [8, 16, 32, 64])
@pytest.mark.parametrize("T", [1, 37, 64, 130])
def test_chunked_equals_recurrence(C, T):
    rng = np.random.default_rng(C * 1000 + T)
    n, dv = 8, 6
    q, k, v, a, b = _inputs(rng, T, n, dv)
    h0 = rng.standard_normal((n, dv))
    o_ref, h_ref = oracle.fwd(q[None, None], k[None, None], v[None, None], a[None, None],
                              b[None, None], h0[None, None])
    o, h = chunked_forward(q, k, v, a, b, h0, C=C)
    scale = max(1.0, np.abs(o_ref).max())
    np.testing.assert_allclose(o, o_ref[0, 0], atol=1e-10 * scale, rtol=0)
    np.testing.assert_allclose(h, h_ref[0, 0], atol=1e-10 * scale, rtol=0)


def test_gated_gram_matches_explicit_products():
    rng = np.random.default_rng(3)
    C, n = 16, 5
    q, k, _, a, _ = _inputs(rng, C, n, 1, zeros=0.2, negs=0.2)
    Gk, Gq = gated_grams(q, k, a)
    for t in range(C):
        for s in range(C):
            g = np.prod(a[s + 1:t + 1], axis=0) if s < t else np.ones(n)
            want_k = np.sum(k[t] * k[s] * g) if s < t else 0.0
            want_q = np.sum(q[t] * k[s] * g) if s <= t else 0.0
            assert abs(Gk[t, s] - want_k) < 1e-13
            assert abs(Gq[t, s] - want_q) < 1e-13


def test_all_zero_gates_and_identity_tail():
    """alpha = 0 everywhere erases the carried state at every token; a chunk
    of pure padding leaves the state untouched."""
    rng = np.random.default_rng(4)
    T, n, dv = 20, 4, 3
    q, k, v, _, b = _inputs(rng, T, n, dv)
    a = np.zeros((T, n))
    h0 = rng.standard_normal((n, dv))
    o_ref, h_ref = oracle.fwd(q[None, None], k[None, None], v[None, None], a[None, None],
                              b[None, None], h0[None, None])
    o, h = chunked_forward(q, k, v, a, b, h0, C=8)
    np.testing.assert_allclose(o, o_ref[0, 0], atol=1e-12)
    np.testing.assert_allclose(h, h_ref[0, 0], atol=1e-12)
