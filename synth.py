"""Seeded synthetic inputs for the CKDA forward and decode workloads.

This module only draws random numbers; it holds none of the recurrence's
arithmetic.  Both the fp64 oracle and the CUDA library consume what it makes,
so it is the one piece they share.

Recipe (every workload):
  * torch CPU generator seeded once per workload; draws happen in fp32, in the
    order lengths (packed only), q, k, v, alpha-source, alpha-masks, beta,
    h0; then each tensor is cast once to the I/O dtype (round to nearest even).
  * q, v ~ N(0, 1).  k ~ N(0, 1), then L2-normalised per token in fp32 (the
    recurrence wants unit keys; the cast to bf16 leaves |k| within ~2^-8 of 1).
  * Gate distributions, by workload family:
      "uniform" : alpha ~ U[-1, 1], beta ~ U[0, 2]
      "kda"     : alpha = sigmoid(N(2, 1)) in (0, 1), beta = sigmoid(N(0, 1))
      "ckda"    : alpha = tanh(N(0, std 2)); then per entry u ~ U[0, 1):
                  u < 0.01 -> 0, 0.01 <= u < 0.11 -> -1;  beta = 2 sigmoid(N(0, 1))
  * h0 ~ N(0, std 0.1) in fp32 when requested, else None (zero state).
  * N(mu, s) means mean mu and standard deviation s.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

# --- the named workloads ------------------------------------------------------

WORKLOADS = {
    "tiny_fp32": dict(B=1, H=1, T=64, d=16, dist="uniform", dtype="fp32", h0=False,
                      seed=0, chunk=16),
    "kda_range": dict(B=8, H=16, T=2048, d=128, dist="kda", dtype="bf16", h0=False,
                      seed=1, chunk=64),
    "ckda_full": dict(B=4, H=32, T=8192, d=128, dist="ckda", dtype="bf16", h0=True,
                      seed=2, chunk=64),
    "ckda_varlen": dict(N=64, H=16, Lmin=128, Lmax=16384, d=128, dist="ckda",
                        dtype="bf16", h0=False, seed=3, chunk=64),
    "ckda_decode": dict(B=256, H=32, d=128, steps=1000, dist="ckda", dtype="bf16",
                        seed=4),
    # the KDA-range forward with the reduced key dimension of a state-reduced
    # head ("On State Reduction in Linear Attention": dk' = 64 of dv = 128)
    "kda_range_dk64": dict(B=8, H=16, T=2048, d=64, dv=128, dist="kda", dtype="bf16",
                           h0=False, seed=5, chunk=64),
    # one long sequence of 16 heads: the paper's Fig. 5 timing shape (16 heads,
    # d = 128, 32k tokens per step) as a single sequence, with the full CKDA
    # gate distribution
    "long_seq": dict(B=1, H=16, T=32768, d=128, dist="ckda", dtype="bf16", h0=True,
                     seed=6, chunk=64),
}

_DT = {"fp32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class FwdInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    alpha: torch.Tensor
    beta: torch.Tensor
    h0: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]  # int32 [N+1] or None

    @property
    def num_seqs(self) -> int:
        return self.q.shape[0] if self.cu_seqlens is None else self.cu_seqlens.numel() - 1

    def to(self, device):
        f = lambda t: None if t is None else t.to(device)
        return FwdInputs(f(self.q), f(self.k), f(self.v), f(self.alpha), f(self.beta),
                         f(self.h0), f(self.cu_seqlens))


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _unit_keys(shape, g):
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    return k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def _gates(shape_a, shape_b, dist, g):
    if dist == "uniform":
        a = torch.rand(shape_a, generator=g) * 2.0 - 1.0
        b = torch.rand(shape_b, generator=g) * 2.0
    elif dist == "kda":
        a = torch.sigmoid(torch.randn(shape_a, generator=g) + 2.0)
        b = torch.sigmoid(torch.randn(shape_b, generator=g))
    elif dist == "ckda":
        a = torch.tanh(torch.randn(shape_a, generator=g) * 2.0)
        u = torch.rand(shape_a, generator=g)
        a = torch.where(u < 0.01, torch.zeros_like(a), a)
        a = torch.where((u >= 0.01) & (u < 0.11), -torch.ones_like(a), a)
        b = 2.0 * torch.sigmoid(torch.randn(shape_b, generator=g))
    else:
        raise ValueError(f"unknown gate distribution {dist!r}")
    return a, b


def make_fwd(B, H, T, dk, dv=None, dist="ckda", dtype="bf16", h0=False, seed=0):
    """Dense [B, H, T, d] inputs."""
    dv = dk if dv is None else dv
    g = _gen(seed)
    q = torch.randn((B, H, T, dk), generator=g)
    k = _unit_keys((B, H, T, dk), g)
    v = torch.randn((B, H, T, dv), generator=g)
    a, b = _gates((B, H, T, dk), (B, H, T), dist, g)
    h = torch.randn((B, H, dk, dv), generator=g) * 0.1 if h0 else None
    dt = _DT[dtype]
    return FwdInputs(q.to(dt), k.to(dt), v.to(dt), a.to(dt), b.to(dt), h, None)


def make_lengths(N, Lmin, Lmax, seed=None, generator=None):
    """N lengths ~ U{Lmin..Lmax} (inclusive)."""
    g = generator if generator is not None else _gen(seed)
    return torch.randint(Lmin, Lmax + 1, (N,), generator=g)


def make_varlen(lengths, H, dk, dv=None, dist="ckda", dtype="bf16", h0=False, seed=0,
                generator=None):
    """Packed variable-length inputs: [1, H, sum(L), d] with cu_seqlens.

    With `generator` given the values continue that generator's stream (the
    named packed workload draws its lengths first from the same stream)."""
    dv = dk if dv is None else dv
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    g = generator if generator is not None else _gen(seed)
    Tt = int(lengths.sum())
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
    q = torch.randn((1, H, Tt, dk), generator=g)
    k = _unit_keys((1, H, Tt, dk), g)
    v = torch.randn((1, H, Tt, dv), generator=g)
    a, b = _gates((1, H, Tt, dk), (1, H, Tt), dist, g)
    h = torch.randn((lengths.numel(), H, dk, dv), generator=g) * 0.1 if h0 else None
    dt = _DT[dtype]
    return FwdInputs(q.to(dt), k.to(dt), v.to(dt), a.to(dt), b.to(dt), h, cu)


def make_workload(name, **override):
    """Inputs of one named workload (optionally with some sizes overridden)."""
    w = dict(WORKLOADS[name])
    w.update(override)
    if name == "ckda_varlen":
        g = _gen(w["seed"])
        lengths = make_lengths(w["N"], w["Lmin"], w["Lmax"], generator=g)
        return make_varlen(lengths, w["H"], w["d"], dist=w["dist"], dtype=w["dtype"],
                           h0=w["h0"], generator=g)
    return make_fwd(w["B"], w["H"], w["T"], w["d"], dv=w.get("dv"), dist=w["dist"],
                    dtype=w["dtype"], h0=w["h0"], seed=w["seed"])


# --- decode -----------------------------------------------------------------

def decode_step_seed(base_seed: int, step: int) -> int:
    """Seed of decode step `step`: the pair (base_seed, step) packed in 64 bits."""
    return (int(base_seed) << 32) | int(step)


def make_decode_state(B, H, dk, dv=None, seed=4):
    dv = dk if dv is None else dv
    g = _gen(seed)
    return torch.randn((B, H, dk, dv), generator=g) * 0.1


def make_decode_step(B, H, dk, dv=None, dist="ckda", dtype="bf16", seed=4, step=0):
    """Single-token inputs of one decode step: q,k,alpha [B,H,dk]; v [B,H,dv]; beta [B,H]."""
    dv = dk if dv is None else dv
    g = _gen(decode_step_seed(seed, step))
    q = torch.randn((B, H, dk), generator=g)
    k = _unit_keys((B, H, dk), g)
    v = torch.randn((B, H, dv), generator=g)
    a, b = _gates((B, H, dk), (B, H), dist, g)
    dt = _DT[dtype]
    return q.to(dt), k.to(dt), v.to(dt), a.to(dt), b.to(dt)
