"""GPU checks of ckda_fwd_host, the forward over host buffers.

Slices of tokens are copied in, computed and copied out on separate streams,
with the state carried between slices in fp32 device memory.  Slices end on
chunk boundaries, so every output must equal ckda_fwd's bit for bit (and
ckda_fwd is checked against the oracle in test_gpu_fwd); one case is also
compared with the oracle directly.
"""
import pytest
import torch

import oracle
import synth
from metrics import report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ck():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_ckda_gb300 as ck
    ck.lib()  # raises if the library is missing: no fallback
    return ck


def host_run(ck, x, slice_tokens, h0_on):
    hq, hk, hv, ha, hb = (t.pin_memory() for t in (x.q, x.k, x.v, x.alpha, x.beta))
    h0 = x.h0.pin_memory() if (h0_on and x.h0 is not None) else None
    o, hT = ck.fwd_host(hq, hk, hv, ha, hb, h0=h0, slice_tokens=slice_tokens)
    st = ck.fwd_status(ck.fwd_host.last_scratch)
    torch.cuda.synchronize()
    assert st == 0, f"device status {ck.STATUS.get(st, st)}"
    return o, hT


def device_run(ck, x, h0_on):
    d = x.to("cuda")
    o, hT = ck.fwd(d.q, d.k, d.v, d.alpha, d.beta, d.h0 if h0_on else None)
    st = ck.fwd_status(ck.fwd.last_workspace)
    torch.cuda.synchronize()
    assert st == 0
    return o.cpu(), hT.cpu()


@pytest.mark.parametrize("T,slice_tokens,h0_on", [
    (300, 128, True),    # slices 128, 128, 44
    (1000, 0, True),     # automatic slice (512), ragged last slice
    (64, 64, False),     # one slice
    (640, 64, False),    # ten one-chunk slices
])
def test_host_equals_device_tensor_path(ck, T, slice_tokens, h0_on):
    x = synth.make_fwd(2, 3, T, 128, dist="ckda", dtype="bf16", h0=True, seed=41)
    o_h, hT_h = host_run(ck, x, slice_tokens, h0_on)
    o_d, hT_d = device_run(ck, x, h0_on)
    assert torch.equal(o_h, o_d)
    assert torch.equal(hT_h, hT_d)


def test_host_equals_device_recurrent_path(ck):
    x = synth.make_fwd(1, 2, 200, 64, dist="ckda", dtype="fp32", h0=True, seed=42)
    o_h, hT_h = host_run(ck, x, 64, True)
    o_d, hT_d = device_run(ck, x, True)
    assert torch.equal(o_h, o_d)
    assert torch.equal(hT_h, hT_d)


def test_host_matches_oracle(ck):
    x = synth.make_fwd(1, 2, 500, 128, dist="ckda", dtype="bf16", h0=True, seed=43)
    o, hT = host_run(ck, x, 128, True)
    o_ref, h_ref = oracle.fwd(x.q, x.k, x.v, x.alpha, x.beta, x.h0)
    ro = report("host o", o, o_ref, True)
    rh = report("host hT", hT, h_ref, False)
    assert ro["excess_bf16"] <= 2e-2 and rh["max_rel"] <= 2e-2


def test_host_empty_sequence_returns_h0(ck):
    x = synth.make_fwd(1, 2, 0, 128, dist="ckda", dtype="bf16", h0=True, seed=44)
    o, hT = host_run(ck, x, 0, True)
    assert o.numel() == 0
    assert torch.equal(hT, x.h0)
