"""The entry points under CUDA graph capture.

A serving loop replays a captured graph instead of launching each call.  The
calls of the hot path enqueue only kernels and asynchronous memsets on the
caller's stream, so they can be captured; these tests capture them and check
that a replay gives bit for bit what the same calls give when launched
directly (the kernels are deterministic).  Parity of the direct calls with the
oracle is the business of the other GPU tests.
"""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ck():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_ckda_gb300 as ck
    ck.lib()
    return ck


def capture(fn):
    """fn() once on a side stream (warm-up), then captured into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("packed", [False, True])
def test_fwd_replay_equals_direct(ck, packed):
    if packed:
        x = synth.make_varlen([70, 1, 300, 0, 129], 3, 128, dist="ckda", dtype="bf16", h0=True,
                              seed=61)
    else:
        x = synth.make_fwd(2, 3, 333, 128, dist="ckda", dtype="bf16", h0=True, seed=61)
    d = x.to("cuda")
    o_ref, h_ref = ck.fwd(d.q, d.k, d.v, d.alpha, d.beta, d.h0, d.cu_seqlens)
    assert ck.fwd_status(ck.fwd.last_workspace) == 0
    o = torch.full_like(o_ref, float("nan"))
    hT = torch.full_like(h_ref, float("nan"))
    wsp = ck.new_workspace(d.num_seqs if d.cu_seqlens is not None else 0, d.q.shape[1],
                           torch.device("cuda"))
    g = capture(lambda: ck.fwd(d.q, d.k, d.v, d.alpha, d.beta, d.h0, d.cu_seqlens, o=o, hT=hT,
                               workspace=wsp))
    o.fill_(float("nan"))
    hT.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert ck.fwd_status(wsp) == 0
    assert torch.equal(o, o_ref) and torch.equal(hT, h_ref)


def test_fwd_split_replay_equals_direct(ck):
    x = synth.make_fwd(1, 2, 1500, 128, dist="kda", dtype="bf16", h0=True, seed=62)
    d = x.to("cuda")
    o_ref, h_ref = ck.fwd_split(d.q, d.k, d.v, d.alpha, d.beta, d.h0, segments=4)
    o = torch.empty_like(o_ref)
    hT = torch.empty_like(h_ref)
    B, H, T, dk = d.q.shape
    wsp = torch.empty(ck.split_workspace_bytes(B, H, T, dk, 128, segments=4), dtype=torch.uint8,
                      device="cuda")
    g = capture(lambda: ck.fwd_split(d.q, d.k, d.v, d.alpha, d.beta, d.h0, segments=4, o=o,
                                     hT=hT, workspace=wsp))
    o.zero_()
    hT.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert ck.fwd_status(wsp) == 0
    assert torch.equal(o, o_ref) and torch.equal(hT, h_ref)


def test_decode_chain_replay_equals_direct(ck):
    B, H, d, steps = 4, 3, 128, 5
    S0 = synth.make_decode_state(B, H, d, seed=63).cuda()
    ins = [tuple(t.cuda() for t in synth.make_decode_step(B, H, d, seed=63, step=i))
           for i in range(steps)]
    S_ref = S0.clone()
    o_ref = [ck.decode_step(*ins[i], S_ref) for i in range(steps)]
    S = S0.clone()
    outs = [torch.empty_like(o_ref[0]) for _ in range(steps)]

    def chain():
        for i in range(steps):
            ck.decode_step(*ins[i], S, o=outs[i])

    g = capture(chain)              # the warm-up and the capture each ran the chain once
    S.copy_(S0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(S, S_ref)
    for a, b in zip(outs, o_ref):
        assert torch.equal(a, b)


def test_fwd_split_varlen_replay_equals_direct(ck):
    x = synth.make_varlen([2000, 100, 0, 700, 64], 2, 128, dist="ckda", dtype="bf16", h0=True,
                          seed=64)
    d = x.to("cuda")
    seg = 512
    o_ref, h_ref = ck.fwd_split_varlen(d.q, d.k, d.v, d.alpha, d.beta, d.cu_seqlens, h0=d.h0,
                                       seg_len=seg)
    o = torch.empty_like(o_ref)
    hT = torch.empty_like(h_ref)
    N, H, T = d.num_seqs, d.q.shape[1], d.q.shape[2]
    wsp = torch.empty(max(256, ck.split_varlen_workspace_bytes(N, H, T, 128, seg)),
                      dtype=torch.uint8, device="cuda")
    g = capture(lambda: ck.fwd_split_varlen(d.q, d.k, d.v, d.alpha, d.beta, d.cu_seqlens,
                                            h0=d.h0, seg_len=seg, o=o, hT=hT, workspace=wsp))
    o.zero_()
    hT.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert ck.fwd_status(wsp) == 0
    assert torch.equal(o, o_ref) and torch.equal(hT, h_ref)


def _randn(shape, seed, dtype=torch.bfloat16, mul=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * mul).to(dtype).cuda()


def test_fwd_raw_replay_equals_direct(ck):
    B, H, T, d = 2, 2, 200, 128
    q, k, a = (_randn((B, H, T, d), 65 + i, mul=3.0) for i in range(3))
    b = _randn((B, H, T), 68)
    v = _randn((B, H, T, d), 69)
    o_ref, h_ref = ck.fwd_raw(q, k, v, a, b)
    o = torch.empty_like(o_ref)
    hT = torch.empty_like(h_ref)
    wsp = ck.new_workspace(0, H, torch.device("cuda"))
    g = capture(lambda: ck.fwd_raw(q, k, v, a, b, o=o, hT=hT, workspace=wsp))
    o.zero_()
    hT.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert ck.fwd_status(wsp) == 0
    assert torch.equal(o, o_ref) and torch.equal(hT, h_ref)


def test_prep_and_prep_bwd_replay_equal_direct(ck):
    rows, d = 300, 128
    q, k, a = (_randn((rows, d), 70 + i, mul=3.0) for i in range(3))
    b = _randn((rows,), 73)
    gq, gk, ga = (_randn((rows, d), 74 + i) for i in range(3))
    gb = _randn((rows,), 77)
    ref_f = ck.prep(k, a, b, q_raw=q)
    ref_b = ck.prep_bwd(k, a, b, gk, ga, gb, q_raw=q, d_q=gq)
    res = []
    g = capture(lambda: res.append((ck.prep(k, a, b, q_raw=q),
                                    ck.prep_bwd(k, a, b, gk, ga, gb, q_raw=q, d_q=gq))))
    out_f, out_b = res[-1]           # the captured call's outputs, from the graph's pool
    for t in out_f + out_b:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for x, y in zip(out_f + out_b, ref_f + ref_b):
        assert torch.equal(x, y)


def test_bwd_replay_equals_direct(ck):
    x = synth.make_fwd(1, 2, 300, 128, dist="ckda", dtype="bf16", h0=True, seed=78)
    d = x.to("cuda")
    do = _randn(tuple(d.v.shape), 79)
    B, H, T, dk = d.q.shape
    wsp = torch.empty(max(16, ck.bwd_workspace_bytes(B, H, T, dk, 128)), dtype=torch.uint8,
                      device="cuda")
    ref = ck.bwd(d.q, d.k, d.v, d.alpha, d.beta, do, h0=d.h0, workspace=wsp)
    res = []
    g = capture(lambda: res.append(ck.bwd(d.q, d.k, d.v, d.alpha, d.beta, do, h0=d.h0,
                                          workspace=wsp)))
    out = res[-1]
    for t in out:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for x_, y in zip(out, ref):
        assert torch.equal(x_, y)


def test_decode_raw_chain_replay_equals_direct(ck):
    B, H, d, steps = 3, 2, 128, 4
    S0 = synth.make_decode_state(B, H, d, seed=80).cuda()
    ins = [(_randn((B, H, d), 81 + 5 * i, mul=3.0), _randn((B, H, d), 82 + 5 * i, mul=2.0),
            _randn((B, H, d), 83 + 5 * i), _randn((B, H, d), 84 + 5 * i, mul=3.0),
            _randn((B, H), 85 + 5 * i)) for i in range(steps)]
    S_ref = S0.clone()
    o_ref = [ck.decode_step_raw(*ins[i], S_ref) for i in range(steps)]
    S = S0.clone()
    outs = [torch.empty_like(o_ref[0]) for _ in range(steps)]

    def chain():
        for i in range(steps):
            ck.decode_step_raw(*ins[i], S, o=outs[i])

    g = capture(chain)
    S.copy_(S0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(S, S_ref)
    for a_, b_ in zip(outs, o_ref):
        assert torch.equal(a_, b_)
