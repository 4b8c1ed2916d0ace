"""GPU parity of ckda_decode_step (C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from metrics import excess_bf16, max_rel, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ck():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_ckda_gb300 as ck
    ck.lib()
    return ck


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("d", [128, 64, 16])
def test_decode_chain_small(ck, dtype, d):
    B, H, steps = 3, 5, 6
    S = synth.make_decode_state(B, H, d, seed=40 + d)
    Sg = S.cuda()
    Sref = S.double().numpy()
    for step in range(steps):
        q, k, v, a, b = synth.make_decode_step(B, H, d, dtype=dtype, seed=40 + d, step=step)
        o = ck.decode_step(q.cuda(), k.cuda(), v.cuda(), a.cuda(), b.cuda(), Sg, scale=0.9)
        o_ref, Sref = oracle.decode_step(q, k, v, a, b, Sref, scale=0.9)
        tol = 2e-2 if dtype == "bf16" else 1e-4
        if dtype == "bf16":
            assert excess_bf16(o.cpu(), o_ref) <= tol
        else:
            assert max_rel(o.cpu(), o_ref) <= tol
        # the state is fp32 throughout: fp32 arithmetic error only
        assert max_rel(Sg.cpu(), Sref) <= 1e-5


def test_decode_workload_full_size(ck):
    """B = 256, H = 32, d = 128: 4 chained steps on the resident state, every
    output and the whole state compared with the oracle."""
    w = synth.WORKLOADS["ckda_decode"]
    B, H, d = w["B"], w["H"], w["d"]
    S = synth.make_decode_state(B, H, d, seed=w["seed"])
    Sg = S.cuda()
    Sref = S.double().numpy()
    for step in range(4):
        q, k, v, a, b = synth.make_decode_step(B, H, d, seed=w["seed"], step=step)
        o = ck.decode_step(q.cuda(), k.cuda(), v.cuda(), a.cuda(), b.cuda(), Sg)
        o_ref, Sref = oracle.decode_step(q, k, v, a, b, Sref)
        r = report(f"decode step {step} o", o.cpu(), o_ref, True)
        assert r["excess_bf16"] <= 2e-2
    assert max_rel(Sg.cpu(), Sref) <= 1e-5


def test_decode_chain_1000_steps(ck):
    """The decode workload's 1000 chained steps on the resident state, at a
    reduced B x H (B = 8, H = 4, d = 128) and the workload's distributions:
    every step's o and the final state against the fp64 oracle, so that fp32
    drift over the whole chain is pinned."""
    w = synth.WORKLOADS["ckda_decode"]
    B, H, d, steps = 8, 4, w["d"], 1000
    S = synth.make_decode_state(B, H, d, seed=w["seed"])
    Sg = S.cuda()
    Sref = S.double().numpy()
    worst = 0.0
    for step in range(steps):
        q, k, v, a, b = synth.make_decode_step(B, H, d, seed=w["seed"], step=step)
        o = ck.decode_step(q.cuda(), k.cuda(), v.cuda(), a.cuda(), b.cuda(), Sg)
        o_ref, Sref = oracle.decode_step(q, k, v, a, b, Sref)
        worst = max(worst, excess_bf16(o.cpu(), o_ref))
    print(f"[decode 1000 steps] worst o excess {worst:.3e}, final state "
          f"{max_rel(Sg.cpu(), Sref):.3e}")
    assert worst <= 2e-2
    assert max_rel(Sg.cpu(), Sref) <= 1e-4


def test_decode_chain_equals_fwd(ck):
    """T decode steps equal one forward over the same T tokens (state and
    outputs), with the token-serial fp32 path on both sides."""
    B, H, d, T = 2, 3, 32, 9
    x = synth.make_fwd(B, H, T, d, dist="ckda", dtype="fp32", h0=True, seed=41)
    d_ = x.to("cuda")
    o_f, h_f = ck.fwd(d_.q, d_.k, d_.v, d_.alpha, d_.beta, d_.h0)
    S = d_.h0.clone()
    for t in range(T):
        o_t = ck.decode_step(d_.q[:, :, t].contiguous(), d_.k[:, :, t].contiguous(),
                             d_.v[:, :, t].contiguous(), d_.alpha[:, :, t].contiguous(),
                             d_.beta[:, :, t].contiguous(), S)
        assert torch.allclose(o_t, o_f[:, :, t], rtol=1e-6, atol=1e-6)
    assert torch.allclose(S, h_f, rtol=1e-6, atol=1e-6)


def raw_step(B, H, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, d), generator=g) * 3
    k = torch.randn((B, H, d), generator=g) * torch.rand((B, H, 1), generator=g) * 5
    v = torch.randn((B, H, d), generator=g)
    a = torch.randn((B, H, d), generator=g) * 3
    b = torch.randn((B, H), generator=g) * 2
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return tuple(t.to(dt) for t in (q, k, v, a, b))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("normalize_q", [True, False])
def test_decode_raw_chain_matches_oracle(ck, dtype, normalize_q):
    """Raw q, k and gate logits through the fused step, against the oracle's
    input preparation followed by the oracle's decode step, 6 chained steps."""
    B, H, d = 3, 5, 128
    S = synth.make_decode_state(B, H, d, seed=70)
    Sg = S.cuda()
    Sref = S.double().numpy()
    for step in range(6):
        q, k, v, a, b = raw_step(B, H, d, dtype, 700 + step)
        o = ck.decode_step_raw(q.cuda(), k.cuda(), v.cuda(), a.cuda(), b.cuda(), Sg, scale=0.8,
                               normalize_q=normalize_q)
        qp, kp, ap, bp = oracle.prep(k, a, b, q_raw=q, normalize_q=normalize_q)
        o_ref, Sref = oracle.decode_step(qp, kp, v, ap, bp, Sref, scale=0.8)
        if dtype == "bf16":
            assert excess_bf16(o.cpu(), o_ref) <= 2e-2
        else:
            assert max_rel(o.cpu(), o_ref) <= 1e-4
        assert max_rel(Sg.cpu(), Sref) <= 1e-5


def test_decode_raw_equals_prep_then_decode(ck):
    """fp32: the fused step equals ckda_prep followed by ckda_decode_step up to
    fp32 rounding (the two sum the norms in different orders)."""
    B, H, d = 4, 6, 128
    S = synth.make_decode_state(B, H, d, seed=71).cuda()
    S2 = S.clone()
    q, k, v, a, b = (t.cuda() for t in raw_step(B, H, d, "fp32", 710))
    o1 = ck.decode_step_raw(q, k, v, a, b, S)
    qp, kp, ap, bp = ck.prep(k, a, b, q_raw=q)
    o2 = ck.decode_step(qp, kp, v, ap, bp, S2)
    assert torch.allclose(o1, o2, rtol=1e-5, atol=1e-6)
    assert torch.allclose(S, S2, rtol=1e-5, atol=1e-6)
