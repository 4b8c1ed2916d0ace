"""GPU parity of ckda_bwd (C ABI) against the fp64 oracle's reverse-mode
gradients, which central differences of the forward oracle pin.

Gradients in the bf16 I/O dtype are held to the forward's bf16 reading (the
error beyond the output's own bf16 rounding, <= 2e-2 of rms, and rms error
<= 5e-3 of rms); fp32 outputs (every gradient with fp32 I/O, and dh0) to
max|err| <= 1e-4 rms.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from metrics import excess_bf16, max_rel, rms_rel

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dalpha", "dbeta", "dh0")


@pytest.fixture(scope="module")
def ck():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_ckda_gb300 as ck
    ck.lib()
    return ck


def grads_case(x, seed, dhT_on=True):
    g = torch.Generator().manual_seed(seed)
    do = torch.randn(x.v.shape, generator=g).to(x.v.dtype)
    N = x.num_seqs
    B, H, T, dk = x.q.shape
    dv = x.v.shape[-1]
    dhT = torch.randn((N, H, dk, dv), generator=g) * 0.5 if dhT_on else None
    return do, dhT


def run(ck, x, do, dhT, scale):
    d = x.to("cuda")
    out = ck.bwd(d.q, d.k, d.v, d.alpha, d.beta, do.cuda(), h0=d.h0,
                 dhT=None if dhT is None else dhT.cuda(), cu_seqlens=d.cu_seqlens, scale=scale)
    torch.cuda.synchronize()
    return [None if t is None else t.cpu() for t in out]


def check(gpu, ref, bf16, name):
    for n, gg, rr in zip(NAMES, gpu, ref):
        if n == "dh0" or not bf16:
            e = max_rel(gg, rr)
            assert e <= 1e-4, (name, n, e)
        else:
            e = excess_bf16(gg, rr)
            assert e <= 2e-2, (name, n, e)
            assert rms_rel(gg, rr) <= 5e-3, (name, n)


@pytest.mark.parametrize("d", [16, 64])
def test_bwd_fp32(ck, d):
    x = synth.make_fwd(2, 2, 77, d, dist="ckda", dtype="fp32", h0=True, seed=500 + d)
    do, dhT = grads_case(x, 600 + d)
    gpu = run(ck, x, do, dhT, 0.7)
    ref = oracle.bwd(x.q, x.k, x.v, x.alpha, x.beta, do, h0=x.h0, dhT=dhT, scale=0.7)
    check(gpu, ref, False, f"fp32 d={d}")


@pytest.mark.parametrize("T", [1, 64, 130])
def test_bwd_bf16_d128(ck, T):
    x = synth.make_fwd(2, 3, T, 128, dist="ckda", dtype="bf16", h0=True, seed=510 + T)
    do, dhT = grads_case(x, 610 + T)
    gpu = run(ck, x, do, dhT, 1.0)
    ref = oracle.bwd(x.q, x.k, x.v, x.alpha, x.beta, do, h0=x.h0, dhT=dhT)
    check(gpu, ref, True, f"bf16 T={T}")


def test_bwd_rectangular_no_h0_no_dhT(ck):
    x = synth.make_fwd(1, 2, 50, 32, dv=48, dist="uniform", dtype="fp32", h0=False, seed=520)
    do, _ = grads_case(x, 620, dhT_on=False)
    gpu = run(ck, x, do, None, 1.0)
    ref = oracle.bwd(x.q, x.k, x.v, x.alpha, x.beta, do)
    check(gpu, ref, False, "dk=32 dv=48")


def test_bwd_partial_column_block(ck):
    """dv = 40: the cluster's third CTA owns 8 live columns of its 16, and
    dk = 24 leaves most row groups inert; T = 201 ends mid-group."""
    x = synth.make_fwd(2, 1, 201, 24, dv=40, dist="ckda", dtype="fp32", h0=True, seed=525)
    do, dhT = grads_case(x, 625)
    gpu = run(ck, x, do, dhT, 0.9)
    ref = oracle.bwd(x.q, x.k, x.v, x.alpha, x.beta, do, h0=x.h0, dhT=dhT, scale=0.9)
    check(gpu, ref, False, "dk=24 dv=40")


def test_bwd_degenerate_gates(ck):
    base = synth.make_fwd(1, 2, 90, 64, dist="ckda", dtype="fp32", h0=True, seed=530)
    do, dhT = grads_case(base, 630)
    for name, a, b in [("alpha0", torch.zeros_like(base.alpha), base.beta),
                       ("alpha-1_beta2", -torch.ones_like(base.alpha),
                        torch.full_like(base.beta, 2.0)),
                       ("beta0", base.alpha, torch.zeros_like(base.beta))]:
        x = synth.FwdInputs(base.q, base.k, base.v, a, b, base.h0, None)
        gpu = run(ck, x, do, dhT, 1.0)
        ref = oracle.bwd(x.q, x.k, x.v, x.alpha, x.beta, do, h0=x.h0, dhT=dhT)
        check(gpu, ref, False, name)


def test_bwd_packed_with_empty_sequences(ck):
    x = synth.make_varlen([0, 1, 65, 0, 30], 2, 128, dist="ckda", dtype="bf16", h0=True,
                          seed=540)
    do, dhT = grads_case(x, 640)
    gpu = run(ck, x, do, dhT, 1.0)
    ref = oracle.bwd(x.q, x.k, x.v, x.alpha, x.beta, do, h0=x.h0, dhT=dhT,
                     cu_seqlens=x.cu_seqlens)
    check(gpu, ref, True, "packed")
    # an empty sequence passes dhT straight through to dh0
    assert torch.equal(gpu[5][0], dhT[0]) and torch.equal(gpu[5][3], dhT[3])


def test_bwd_kda_range_workload_sampled(ck):
    """The KDA-range workload at full size on the GPU; the oracle on two (batch,
    head) units of it (the backward's units are independent)."""
    x = synth.make_workload("kda_range")
    do, _ = grads_case(x, 650, dhT_on=False)
    gpu = run(ck, x, do, None, 1.0)
    for b, h in ((0, 0), (7, 15)):
        sl = lambda t: t[b:b + 1, h:h + 1]
        ref = oracle.bwd(sl(x.q), sl(x.k), sl(x.v), sl(x.alpha), sl(x.beta), sl(do))
        got = [g[b:b + 1, h:h + 1] for g in gpu[:5]] + [gpu[5][b:b + 1, h:h + 1]]
        check(got, ref, True, f"kda_range b={b} h={h}")


def test_bwd_ckda_varlen_workload_sampled(ck):
    """The packed workload at full size (64 sequences, 8.26 M token-heads) on
    the GPU; the oracle, which keeps every state of a pair, on the three
    shortest sequences (their gradients, and dh0 through dhT = 0)."""
    x = synth.make_workload("ckda_varlen")
    do, _ = grads_case(x, 660, dhT_on=False)
    gpu = run(ck, x, do, None, 1.0)
    cu = x.cu_seqlens.numpy()
    lens = np.diff(cu)
    for s in np.argsort(lens, kind="stable")[:3]:
        a0, b0 = int(cu[s]), int(cu[s + 1])
        sl = lambda t: t[:, :, a0:b0]
        ref = oracle.bwd(sl(x.q), sl(x.k), sl(x.v), sl(x.alpha), sl(x.beta), sl(do))
        got = [g[:, :, a0:b0] for g in gpu[:5]] + [gpu[5][s:s + 1]]
        check(got, ref, True, f"varlen seq {s} L={b0 - a0}")
