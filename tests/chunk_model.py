"""fp64 numpy model of the chunkwise algorithm the CUDA forward kernel runs.

This is a test helper, not an oracle: it restates, in plain numpy, the
division-free WY/UT chunk decomposition that the tensor-core kernel uses, so a
test can check that the algebra reaches the token-by-token recurrence exactly
(up to rounding order), including gates that are exactly 0 or -1.

For a chunk of C tokens with chunk-local state H (n x dv), gates alpha_t,
Gamma(t<-s) = prod_{r=s+1..t} alpha_r (per channel; Gamma(t<-t) = 1):

  gamma_t = Gamma(t<-0)          inclusive prefix product
  rho_s   = Gamma(C<-s)          exclusive suffix product
  M[t,s]  = beta_t sum_i k_ti k_si Gamma(t<-s)_i   (s < t)
  A[t,s]  = sum_i q_ti k_si Gamma(t<-s)_i          (s <= t)
  T       = (I + M)^-1
  W       = T Diag(beta) (k * gamma),   Ut = T Diag(beta) V
  U       = Ut - W H
  O       = (q * gamma) H + A U
  H'      = Diag(gamma_C) H + (k * rho)^T U

Gamma(t<-s) is never formed as a ratio.  The strictly-lower pairs are split by
a binary tree over the chunk: a pair (t, s) whose positions first differ at
bit l lies in one aligned segment of 2L = 2^(l+1) tokens, s in its lower and
t in its upper half; with m the last position of the lower half,
Gamma(t<-s) = [prod_{m<r<=t} alpha_r] [prod_{s<r<=m} alpha_r], a forward
product times a backward product, so each level is one dense contraction of
gated operands.  The diagonal of A is q_t . k_t.
"""
import numpy as np


def tree_levels(C):
    L = C // 2
    while L >= 1:
        yield L
        L //= 2


def gated_grams(q, k, alpha):
    """Returns (Gk, Gq): Gk[t,s] = sum_i k_t k_s Gamma(t<-s) for s < t,
    Gq[t,s] = sum_i q_t k_s Gamma(t<-s) for s <= t (zero elsewhere)."""
    C, n = k.shape
    Gk = np.zeros((C, C))
    Gq = np.zeros((C, C))
    for L in tree_levels(C):
        for seg in range(0, C, 2 * L):
            m = seg + L - 1
            f = np.cumprod(alpha[m + 1:m + 1 + L], axis=0)           # t = m+1..m+L
            b = np.ones((L, n))                                       # s = seg..m
            for j in range(L - 2, -1, -1):
                b[j] = b[j + 1] * alpha[seg + j + 1]
            up = slice(m + 1, m + 1 + L)
            lo = slice(seg, m + 1)
            ks = k[lo] * b
            Gk[up, lo] = (k[up] * f) @ ks.T
            Gq[up, lo] = (q[up] * f) @ ks.T
    Gq[np.arange(C), np.arange(C)] = np.einsum("ti,ti->t", q, k)
    return Gk, Gq


def chunk_step(H, q, k, v, alpha, beta, rnd=None):
    """One chunk.  q, k, alpha: [C, n]; v: [C, dv]; beta: [C].  `rnd(name, x)`
    optionally rounds intermediate operands (to model the kernel's storage
    precisions); identity by default."""
    r = rnd or (lambda name, x: x)
    C, n = k.shape
    gamma = np.cumprod(alpha, axis=0)
    rho = np.ones((C, n))
    for s in range(C - 2, -1, -1):
        rho[s] = rho[s + 1] * alpha[s + 1]
    Gk, Gq = gated_grams(q, k, alpha)
    M = beta[:, None] * Gk
    Aqk = r("Aqk", Gq)
    T = np.linalg.inv(np.eye(C) + M)
    TB = r("TB", T * beta[None, :])
    W = r("W", TB @ r("Kg", k * gamma))
    Ut = TB @ v
    Hb = r("H", H)
    U = r("U", Ut - W @ Hb)
    O = r("Qg", q * gamma) @ Hb + Aqk @ U
    Hn = gamma[-1][:, None] * H + r("Kh", k * rho).T @ U
    return O, Hn


def chunked_forward(q, k, v, alpha, beta, h0=None, C=64, rnd=None):
    """Single (sequence, head): q, k, alpha [T, n], v [T, dv], beta [T].
    The tail chunk is padded with identity transitions (alpha = 1, beta = 0)."""
    T, n = k.shape
    dv = v.shape[1]
    H = np.zeros((n, dv)) if h0 is None else np.array(h0, dtype=np.float64)
    O = np.zeros((T, dv))
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        pad = lambda x, fill: np.concatenate([x[c0:c0 + L], np.full((C - L,) + x.shape[1:], fill)])
        Oc, H = chunk_step(H, pad(q, 0.0), pad(k, 0.0), pad(v, 0.0), pad(alpha, 1.0),
                           pad(beta, 0.0), rnd)
        O[c0:c0 + L] = Oc[:L]
    return O, H
