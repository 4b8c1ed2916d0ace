"""Storage precisions for a chunkwise tensor-core backward, chosen by
simulation against the fp64 oracle before any such kernel exists.  The plan
is checked at 256 tokens (4 chunks) and at 2048 (32 chunks, the KDA-range
sequence length), so that errors carried back through the chunks are covered.

The chunk model's rounding hooks round every contraction operand as a kernel
would store it; accumulation stays exact (fp32 in a kernel, whose error is far
below these roundings).  The forward's operands are rounded as the forward
kernel stores them: the gated Grams, W, H, U, q*gamma and k*rho in fp16, and
T Diag(beta) and k*gamma in bf16.  The backward's operands are in fp16.  At
the workloads' shape (d = 128, chunk 64) and gate distributions, every
gradient stays within the bf16 bound, max |err| / rms(ref) <= 2e-2, with a
factor of two to spare.  The same plan with the Gram-gradient operands in bf16
is several times worse, which is why they are fp16.
"""
import numpy as np
import pytest

import chunk_model as cm
import oracle


def bf16(x):
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def fp16(x):
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


FWD = {"Aqk": fp16, "W": fp16, "H": fp16, "U": fp16, "Qg": fp16, "Kh": fp16,
       "TB": bf16, "Kg": bf16}


def plan(overrides):
    def rnd(name, x):
        if name in overrides:
            return overrides[name](x)
        return FWD.get(name, fp16)(x)
    return rnd


def inputs(dist, T=256, n=128, dv=128, seed=7):
    """One head of a workload's distribution (see synth.py), cast to bf16."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, n))
    v = rng.standard_normal((T, dv))
    k = rng.standard_normal((T, n))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    if dist == "kda":
        a = 1 / (1 + np.exp(-(2 + rng.standard_normal((T, n)))))
        b = 1 / (1 + np.exp(-rng.standard_normal(T)))
        h0 = np.zeros((n, dv))
    else:
        a = np.tanh(2 * rng.standard_normal((T, n)))
        u = rng.random((T, n))
        a[u < 0.01] = 0.0
        a[(u >= 0.01) & (u < 0.11)] = -1.0
        b = 2 / (1 + np.exp(-rng.standard_normal(T)))
        h0 = 0.1 * rng.standard_normal((n, dv))
    dO = rng.standard_normal((T, dv))
    q, k, v, a, b, dO = (bf16(x) for x in (q, k, v, a, b, dO))
    return q, k, v, a, b, dO, h0


def errors(x, rnd):
    q, k, v, a, b, dO, h0 = x
    got = cm.chunked_backward(q, k, v, a, b, dO, h0=h0, C=64, rnd=rnd)
    X = lambda z: z[None, None]
    ref = oracle.bwd(X(q), X(k), X(v), X(a), X(b), X(dO), h0=X(h0))
    out = []
    for g, r in zip(got, ref):
        r = np.asarray(r)[0, 0]
        rms = np.sqrt(np.mean(r * r))
        out.append((np.max(np.abs(g - r)) / rms, np.sqrt(np.mean((g - r) ** 2)) / rms))
    return out


@pytest.mark.parametrize("T", [256, 2048])
@pytest.mark.parametrize("dist", ["kda", "ckda"])
def test_fp16_operands_meet_the_bound(dist, T):
    # 4 and 32 chunks: errors carried back through the reverse dH chain over
    # a workload-length sequence stay within the same bound
    for name, (mx, rm) in zip(("dq", "dk", "dv", "dalpha", "dbeta", "dh0"),
                              errors(inputs(dist, T=T), plan({}))):
        assert mx <= 1e-2 and rm <= 1e-3, (dist, T, name, mx, rm)


@pytest.mark.parametrize("dist", ["kda", "ckda"])
def test_bf16_gram_gradient_operands_are_worse(dist):
    x = inputs(dist)
    e16 = errors(x, plan({}))
    e_bf = errors(x, plan({"dG": bf16, "gop": bf16}))
    for i in (0, 1, 3):   # dq, dk, dalpha go through the Gram gradients
        assert e_bf[i][0] >= 2 * e16[i][0], (dist, i, e_bf[i][0], e16[i][0])
