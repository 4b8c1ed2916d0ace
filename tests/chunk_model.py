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


# --- the chunkwise backward -----------------------------------------------------
#
# Reverse mode through chunk_step, in the same algebra.  Given dO (C x dv) and
# dH' (n x dv):
#
#   dU  = A^T dO + (k*rho) dH'             dA = dO U^T (lower, with diagonal)
#   dH  = (q*gamma)^T dO + Diag(gamma_C) dH' - W^T dU
#   dW  = -dU H^T,  dTB = dU V^T + dW (k*gamma)^T,  dV = TB^T dU
#   dT  = dTB Diag(beta),  dM = -T^T dT T^T (strictly lower)
#   dbeta_s += sum_t dTB_ts T_ts,  dbeta_t += sum_s dM_ts Gk_ts
#
# and the gated Grams' transposed products for dk and dq, on the same split
# tree as the forward (gated_grams_bwd).  Every gate gradient is formed
# without division.  For a product chain
# P_t = prod_{r<=t} alpha_r with adjoints g_t:
#   dalpha_r = [prod_{r'<r} alpha_r'] S_r,  with S_r = g_r + alpha_{r+1} S_{r+1}
# (a backward scan), and likewise for the suffix products rho with a forward
# scan.  On the tree, each level's F and B are such chains.


def _pair_products(alpha):
    """G[t, s] = Gamma(t<-s) = prod_{s<r<=t} alpha_r for s <= t (ones on the
    diagonal), built by multiplication along each row."""
    C, n = alpha.shape
    G = np.zeros((C, C, n))
    for s in range(C):
        G[s, s] = 1.0
        for t in range(s + 1, C):
            G[t, s] = G[t - 1, s] * alpha[t]
    return G


def chunk_step_bwd(H, q, k, v, alpha, beta, dO, dHn, rnd=None):
    """Gradients through chunk_step: returns (dH, dq, dk, dv, dalpha, dbeta).
    `rnd(name, x)` optionally rounds the operands of each contraction (to model
    a kernel's storage precisions); identity by default."""
    rd = rnd or (lambda name, x: x)
    C, n = k.shape
    low = np.tril(np.ones((C, C)), -1)              # s < t
    lowd = np.tril(np.ones((C, C)))                 # s <= t
    gamma = np.cumprod(alpha, axis=0)
    rho = np.ones((C, n))
    for s in range(C - 2, -1, -1):
        rho[s] = rho[s + 1] * alpha[s + 1]
    Gk, Gq = gated_grams(q, k, alpha)
    M = beta[:, None] * Gk
    T = np.linalg.inv(np.eye(C) + M)
    TB = rd("TB", T * beta[None, :])
    Tr = rd("T", T)
    Kg, Qg, Kh = rd("Kg", k * gamma), rd("Qg", q * gamma), rd("Kh", k * rho)
    A = rd("A", Gq)
    W = rd("W", TB @ Kg)
    Hr = rd("H", H)
    U = rd("U", TB @ v - W @ Hr)
    dOr, dHr = rd("dO", dO), rd("dHn", dHn)
    # outputs and the next state
    dU = rd("dU", A.T @ dOr + Kh @ dHr)
    dGq = rd("dG", (dOr @ U.T) * lowd)
    dQg = dOr @ Hr.T
    dH = Qg.T @ dOr + gamma[-1][:, None] * dHn - W.T @ dU
    dgC = np.einsum("ij,ij->i", dHn, H)
    dKh = U @ dHr.T
    # the UT/WY transform
    dW = rd("dW", -dU @ Hr.T)
    dTB = dU @ v.T + dW @ Kg.T
    dv = TB.T @ dU
    dKg = TB.T @ dW
    dT = rd("dT", dTB * beta[None, :])
    dbeta = np.einsum("ts,ts->s", dTB, T)
    dM = (-Tr.T @ dT @ Tr.T) * low
    dbeta = dbeta + np.einsum("ts,ts->t", dM, Gk)
    dGk = rd("dG", beta[:, None] * dM)
    # the gated Grams, on the split tree
    dq, dk, dalpha = gated_grams_bwd(q, k, alpha, dGk, dGq, rnd=rnd)
    dq = dq + dQg * gamma
    dk = dk + dKg * gamma + dKh * rho
    # gate gradients of the prefix and suffix products, without division
    dgamma = dKg * k + dQg * q
    dgamma[-1] += dgC                               # gamma_C = gamma_{C-1}
    drho = dKh * k
    S = np.zeros(n)                                 # backward scan over dgamma
    for r in range(C - 1, -1, -1):
        S = dgamma[r] + (alpha[r + 1] * S if r + 1 < C else 0.0)
        dalpha[r] += (gamma[r - 1] if r > 0 else 1.0) * S
    R = np.zeros(n)                                 # forward scan over drho
    for r in range(1, C):
        R = drho[r - 1] + alpha[r - 1] * R if r > 1 else drho[0]
        dalpha[r] += rho[r] * R
    return dH, dq, dk, dv, dalpha, dbeta


def gated_grams_bwd_direct(q, k, alpha, dGk, dGq):
    """The same gradients as gated_grams_bwd from the explicit pair products:
    the factor of alpha_r in Gamma(t<-s), s < r <= t, is Gamma(t<-r)
    Gamma(r-1<-s).  O(C^3 n); a cross-check of the tree form."""
    C, n = k.shape
    G = _pair_products(alpha)
    low = np.tril(np.ones((C, C)), -1)
    dq = np.einsum("ts,si,tsi->ti", dGq, k, G)
    dk = (np.einsum("ts,si,tsi->ti", dGk, k, G) + np.einsum("ts,ti,tsi->si", dGk, k, G)
          + np.einsum("ts,ti,tsi->si", dGq, q, G))
    dG = np.einsum("ts,ti,si->tsi", dGk, k, k) + np.einsum("ts,ti,si->tsi", dGq * low, q, k)
    dalpha = np.zeros((C, n))
    for r in range(1, C):
        for t in range(r, C):
            for s in range(r):
                dalpha[r] += dG[t, s] * G[t, r] * G[r - 1, s]
    return dq, dk, dalpha


def chunked_backward(q, k, v, alpha, beta, dO, h0=None, dhT=None, C=16, rnd=None):
    """Single (sequence, head) backward by chunks: the forward keeps the state
    at each chunk start, then the chunks run in reverse through
    chunk_step_bwd.  Returns (dq, dk, dv, dalpha, dbeta, dh0)."""
    T, n = k.shape
    dvn = v.shape[1]
    H = np.zeros((n, dvn)) if h0 is None else np.array(h0, dtype=np.float64)

    def pad(x, c0, L, fill):
        return np.concatenate([x[c0:c0 + L], np.full((C - L,) + x.shape[1:], fill)])

    starts = []
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        starts.append(H)
        _, H = chunk_step(H, pad(q, c0, L, 0.0), pad(k, c0, L, 0.0), pad(v, c0, L, 0.0),
                          pad(alpha, c0, L, 1.0), pad(beta, c0, L, 0.0), rnd)
    dH = np.zeros((n, dvn)) if dhT is None else np.array(dhT, dtype=np.float64)
    out = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(alpha),
           np.zeros_like(beta)]
    for ci in range(len(starts) - 1, -1, -1):
        c0 = ci * C
        L = min(C, T - c0)
        dH, *g = chunk_step_bwd(starts[ci], pad(q, c0, L, 0.0), pad(k, c0, L, 0.0),
                                pad(v, c0, L, 0.0), pad(alpha, c0, L, 1.0),
                                pad(beta, c0, L, 0.0), pad(dO, c0, L, 0.0), dH, rnd)
        for o, gg in zip(out, g):
            o[c0:c0 + L] = gg[:L]
    return (*out, dH)


def gated_grams_bwd(q, k, alpha, dGk, dGq, rnd=None):
    """Gradients of the gated Grams (Gk strictly lower, Gq lower with diagonal)
    on the split tree the forward uses: on each level, Gamma(t<-s) = F_t B_s with
    F_t = prod_{m<r<=t} alpha_r over the upper half and B_s = prod_{s<r<=m}
    alpha_r over the lower half.  Per level and segment:
      d(k F)_t = dGk[t, :] (k B),   d(q F)_t = dGq[t, :] (k B)     (upper rows)
      d(k B)_s = dGk[:, s]^T (k F) + dGq[:, s]^T (q F)             (lower rows)
    then dk, dq by the factors, and dalpha from F by a backward scan and from
    B by a forward scan.  Returns (dq, dk, dalpha).  `rnd` as in chunk_step_bwd
    (the gated operands are "gop")."""
    rd = rnd or (lambda name, x: x)
    C, n = k.shape
    dq = np.zeros((C, n))
    dk = np.zeros((C, n))
    dalpha = np.zeros((C, n))
    for L in tree_levels(C):
        for seg in range(0, C, 2 * L):
            m = seg + L - 1
            up = slice(m + 1, m + 1 + L)
            lo = slice(seg, m + 1)
            F = np.cumprod(alpha[up], axis=0)
            B = np.ones((L, n))
            for j in range(L - 2, -1, -1):
                B[j] = B[j + 1] * alpha[seg + j + 1]
            kF, qF, kB = rd("gop", k[up] * F), rd("gop", q[up] * F), rd("gop", k[lo] * B)
            dkF = dGk[up, lo] @ kB
            dqF = dGq[up, lo] @ kB
            dkB = dGk[up, lo].T @ kF + dGq[up, lo].T @ qF
            dk[up] += dkF * F
            dq[up] += dqF * F
            dk[lo] += dkB * B
            dF = dkF * k[up] + dqF * q[up]
            dB = dkB * k[lo]
            # F_t = prod_{m<r<=t} alpha_r: dalpha_r = [prod_{m<r'<r}] S_r,
            # S_r = dF_r + alpha_{r+1} S_{r+1}
            S = np.zeros(n)
            for jr in range(L - 1, -1, -1):
                r = m + 1 + jr
                S = dF[jr] + (alpha[r + 1] * S if jr + 1 < L else 0.0)
                dalpha[r] += (F[jr - 1] if jr > 0 else 1.0) * S
            # B_s = prod_{s<r<=m} alpha_r: dalpha_r = [prod_{r<r'<=m}] R_r,
            # R_r = dB_{r-1} + alpha_{r-1} R_{r-1}
            R = np.zeros(n)
            for jr in range(1, L):
                r = seg + jr
                R = dB[jr - 1] + (alpha[r - 1] * R if jr > 1 else 0.0)
                dalpha[r] += B[jr] * R
    # the diagonal of Gq carries no gate
    dq += np.diagonal(dGq)[:, None] * k
    dk += np.diagonal(dGq)[:, None] * q
    return dq, dk, dalpha
