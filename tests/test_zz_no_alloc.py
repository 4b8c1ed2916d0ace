"""ckda_fwd_noalloc, the forward for callers that cannot allocate device
memory, gives the same results as ckda_fwd.

The file is named to be collected last.  If it fails, a run that stops at the
first failure has already run every other test.  It must also pass alone in a
fresh process, where its first call sets up the library's scratch array.
"""
import ctypes

import pytest
import torch

import synth
from metrics import excess_bf16, max_rel

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module")
def ck():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_ckda_gb300 as ck
    ck.lib()
    return ck


def _reference(ck, d):
    o, hT = ck.fwd(d.q, d.k, d.v, d.alpha, d.beta, d.h0, d.cu_seqlens)
    assert ck.fwd_status(ck.fwd.last_workspace) == 0
    return o, hT


def test_noalloc_matches_fwd_two_calls_in_a_row(ck):
    dense = synth.make_fwd(2, 3, 200, 128, dist="ckda", dtype="bf16", h0=True, seed=900).to("cuda")
    packed = synth.make_varlen([70, 1, 0, 129, 64], 2, 128, dist="ckda", dtype="bf16", h0=True,
                               seed=901).to("cuda")
    outs = []
    # two calls in a row on the shared scratch, each compared with ckda_fwd
    for d in (packed, dense):
        o, hT = ck.fwd_noalloc(d.q, d.k, d.v, d.alpha, d.beta, d.h0, d.cu_seqlens)
        torch.cuda.synchronize()
        outs.append((d, o.clone(), hT.clone()))
    for d, o, hT in outs:
        o_ref, h_ref = _reference(ck, d)
        assert excess_bf16(o.cpu(), o_ref.cpu().double()) <= TOL_BF16
        assert max_rel(hT.cpu(), h_ref.cpu()) <= TOL_BF16


def test_noalloc_rejects_too_many_sequences(ck):
    # real (small) device buffers everywhere: if the host-side limit ever
    # stopped rejecting this call, the launch would still only touch valid
    # memory and the assert, not the GPU, would report it
    L = ck.lib()
    n = 65537
    d = synth.make_varlen([1, 2], 1, 128, dist="ckda", dtype="bf16", h0=False, seed=902).to("cuda")
    cu = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
    cu[-1] = d.q.shape[2]
    cu[-2] = d.q.shape[2]
    o = torch.empty_like(d.v)
    vp = ctypes.c_void_p
    L.ckda_fwd_noalloc.argtypes = [vp] * 9 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int, vp]
    L.ckda_fwd_noalloc.restype = ctypes.c_int
    p = lambda t: vp(t.data_ptr())
    rc = L.ckda_fwd_noalloc(p(d.q), p(d.k), p(d.v), p(d.alpha), p(d.beta), None, p(o), None,
                            p(cu), n, 1, 1, d.q.shape[2], 128, 128, 1, 1.0, 0, None)
    torch.cuda.synchronize()
    assert rc == 2  # CKDA_ERR_UNSUPPORTED, nothing launched
