"""GPU parity of ckda_fwd_split and ckda_fwd_split_varlen (C ABI) against the
fp64 oracle.

The sequence split must give the result of one pass over each whole
sequence: o and the final state are compared with the oracle's plain
recurrence for several segment counts, ragged tails, with and without h0,
hT aliasing h0, the 64-wide key, v and h0 far from unit scale, more CTAs
than SMs, and the one-long-sequence workload at full size with the
automatic segment count; for packed input, sequences of 1 to 23 segments
(ragged, empty, one chunk) in one call, the unsplit case against ckda_fwd bit
for bit, dk = 64, scaled inputs, and one long sequence among short ones.
"""
import dataclasses

import pytest
import torch

import oracle
import synth
from metrics import report

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module")
def ck():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_ckda_gb300 as ck
    ck.lib()  # raises if the library is missing: no fallback
    return ck


def run_split(ck, x, segments, h0_on=True, alias=False):
    d = x.to("cuda")
    h0 = d.h0 if h0_on else None
    if alias:
        h0 = h0.clone()
        o, hT = ck.fwd_split(d.q, d.k, d.v, d.alpha, d.beta, h0, segments=segments, hT=h0)
    else:
        o, hT = ck.fwd_split(d.q, d.k, d.v, d.alpha, d.beta, h0, segments=segments)
    st = ck.fwd_status(ck.fwd_split.last_workspace)
    torch.cuda.synchronize()
    assert st == 0, f"device status {ck.STATUS.get(st, st)}"
    return o.cpu(), hT.cpu()


def check(o, hT, x, name, h0_on=True):
    o_ref, h_ref = oracle.fwd(x.q, x.k, x.v, x.alpha, x.beta, x.h0 if h0_on else None)
    ro = report(name + " o", o, o_ref, True)
    rh = report(name + " hT", hT, h_ref, False)
    assert ro["excess_bf16"] <= TOL_BF16, ro
    assert ro["rms_rel"] <= 5e-3, ro
    assert rh["max_rel"] <= TOL_BF16, rh


@pytest.mark.parametrize("segments", [2, 3, 5, 16])
def test_split_matches_oracle(ck, segments):
    # 12 chunks with a ragged tail of 23 tokens; 16 requested -> 12 segments
    x = synth.make_fwd(1, 3, 64 * 11 + 23, 128, dist="ckda", dtype="bf16", h0=True, seed=40)
    o, hT = run_split(ck, x, segments)
    check(o, hT, x, f"split S={segments}")


def test_split_zero_h0_and_batch(ck):
    x = synth.make_fwd(2, 2, 1000, 128, dist="uniform", dtype="bf16", h0=False, seed=41)
    o, hT = run_split(ck, x, 4, h0_on=False)
    check(o, hT, x, "split B=2 zero h0", h0_on=False)


def test_split_hT_aliases_h0(ck):
    x = synth.make_fwd(1, 2, 900, 128, dist="ckda", dtype="bf16", h0=True, seed=42)
    o, hT = run_split(ck, x, 3, alias=True)
    check(o, hT, x, "split hT = h0")


def test_split_dk64(ck):
    x = synth.make_fwd(2, 2, 700, 64, dv=128, dist="kda", dtype="bf16", h0=True, seed=43)
    o, hT = run_split(ck, x, 4)
    check(o, hT, x, "split dk64")


@pytest.mark.parametrize("fv,fh", [(1e6, 1e3), (1e-6, 1.0), (1.0, 1e6)])
def test_split_scaled_inputs(ck, fv, fh):
    """Every pass (from h0, from zero, the transition from [I | 0] with v = 0,
    and from the scanned states) keeps its own power-of-two operand scale."""
    x = synth.make_fwd(1, 2, 64 * 9 + 5, 128, dist="ckda", dtype="bf16", h0=True, seed=45)
    x = dataclasses.replace(x, v=(x.v.float() * fv).to(x.v.dtype), h0=x.h0 * fh)
    o, hT = run_split(ck, x, 4)
    check(o, hT, x, f"split v*{fv:g} h0*{fh:g}")


def test_split_one_segment_is_ckda_fwd(ck):
    """segments = 1 is ckda_fwd itself: the same bits."""
    x = synth.make_fwd(1, 2, 500, 128, dist="ckda", dtype="bf16", h0=True, seed=44)
    d = x.to("cuda")
    o1, h1 = ck.fwd_split(d.q, d.k, d.v, d.alpha, d.beta, d.h0, segments=1)
    o2, h2 = ck.fwd(d.q, d.k, d.v, d.alpha, d.beta, d.h0)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_split_more_ctas_than_sms(ck):
    """KDA-range (128 sequence-heads) forced to 3 segments: 640 CTAs in pass 1."""
    x = synth.make_workload("kda_range")
    o, hT = run_split(ck, x, 3, h0_on=False)
    check(o, hT, x, "split kda_range S=3", h0_on=False)


def test_split_long_seq_workload_full(ck):
    """One sequence of 32768 tokens and 16 heads, with h0, at the automatic
    segment count (the launch configuration the benchmark times)."""
    x = synth.make_workload("long_seq")
    B, H, T, dk = x.q.shape
    S = ck.split_segments(B, H, T, dk, 128)
    assert S >= 3, S
    o, hT = run_split(ck, x, 0)
    check(o, hT, x, f"split long_seq S={S}")


# ------------------------------------------------------------------ packed
def run_split_varlen(ck, x, seg_len, h0_on=True):
    d = x.to("cuda")
    o, hT = ck.fwd_split_varlen(d.q, d.k, d.v, d.alpha, d.beta, d.cu_seqlens,
                                h0=d.h0 if h0_on else None, seg_len=seg_len)
    st = ck.fwd_status(ck.fwd_split_varlen.last_workspace)
    torch.cuda.synchronize()
    assert st == 0, f"device status {ck.STATUS.get(st, st)}"
    return o.cpu(), hT.cpu()


def check_packed(o, hT, x, name, seqs=None, h0_on=True):
    o_ref, h_ref = oracle.fwd(x.q, x.k, x.v, x.alpha, x.beta, x.h0 if h0_on else None,
                              cu_seqlens=x.cu_seqlens)
    cu = x.cu_seqlens.tolist()
    for i in (range(len(cu) - 1) if seqs is None else seqs):
        sl = slice(cu[i], cu[i + 1])
        if cu[i + 1] > cu[i]:
            ro = report(f"{name} seq {i} o", o[:, :, sl], o_ref[:, :, sl], True)
            assert ro["excess_bf16"] <= TOL_BF16 and ro["rms_rel"] <= 5e-3, ro
        rh = report(f"{name} seq {i} hT", hT[i], h_ref[i], False)
        assert rh["max_rel"] <= TOL_BF16, rh


@pytest.mark.parametrize("seg_len", [128, 256, 1024])
def test_split_varlen_matches_oracle(ck, seg_len):
    """Sequences of 1 to 23 segments (ragged ends, an empty one, one of exactly
    one chunk) in one packed call, each against its own oracle run."""
    lengths = [3000, 70, 0, 1500, 64, 129, 700, 2048]
    x = synth.make_varlen(lengths, 2, 128, dist="ckda", dtype="bf16", h0=True, seed=50)
    o, hT = run_split_varlen(ck, x, seg_len)
    check_packed(o, hT, x, f"varlen split {seg_len}")


def test_split_varlen_unsplit_is_ckda_fwd(ck):
    """With every sequence shorter than seg_len nothing is split: the same bits
    as ckda_fwd on the packed input."""
    x = synth.make_varlen([300, 64, 1, 250], 3, 128, dist="ckda", dtype="bf16", h0=True,
                          seed=51)
    d = x.to("cuda")
    o1, h1 = ck.fwd_split_varlen(d.q, d.k, d.v, d.alpha, d.beta, d.cu_seqlens, h0=d.h0,
                                 seg_len=512)
    o2, h2 = ck.fwd(d.q, d.k, d.v, d.alpha, d.beta, d.h0, d.cu_seqlens)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_split_varlen_dk64_zero_h0_and_scaled(ck):
    x = synth.make_varlen([1100, 33, 640], 2, 64, dv=128, dist="kda", dtype="bf16", h0=False,
                          seed=52)
    o, hT = run_split_varlen(ck, x, 256, h0_on=False)
    check_packed(o, hT, x, "varlen split dk64", h0_on=False)
    x = synth.make_varlen([1300, 200], 2, 128, dist="ckda", dtype="bf16", h0=True, seed=53)
    x = dataclasses.replace(x, v=(x.v.float() * 1e6).to(x.v.dtype), h0=x.h0 * 1e3)
    o, hT = run_split_varlen(ck, x, 192)
    check_packed(o, hT, x, "varlen split scaled")


def test_split_varlen_long_tail_workload(ck):
    """One 32k-token sequence packed with 63 of 1k tokens, 16 heads, at the
    automatic segment length: the long one and three short ones against the
    oracle."""
    lengths = [1024] * 31 + [32768] + [1024] * 32
    x = synth.make_varlen(lengths, 16, 128, dist="kda", dtype="bf16", h0=True, seed=54)
    o, hT = run_split_varlen(ck, x, 0)
    sub = [31, 0, 40, 63]
    cu = x.cu_seqlens.tolist()
    for i in sub:
        sl = slice(cu[i], cu[i + 1])
        xi = synth.FwdInputs(x.q[:, :, sl], x.k[:, :, sl], x.v[:, :, sl], x.alpha[:, :, sl],
                             x.beta[:, :, sl], x.h0[i:i + 1], None)
        o_ref, h_ref = oracle.fwd(xi.q, xi.k, xi.v, xi.alpha, xi.beta, xi.h0)
        ro = report(f"long tail seq {i} o", o[:, :, sl], o_ref, True)
        assert ro["excess_bf16"] <= TOL_BF16 and ro["rms_rel"] <= 5e-3, ro
        rh = report(f"long tail seq {i} hT", hT[i:i + 1], h_ref, False)
        assert rh["max_rel"] <= TOL_BF16, rh
