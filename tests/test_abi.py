"""Host-only checks of the C ABI: the library loads, exports every function
include/ckda.h declares, and rejects bad arguments before launching anything.
No call here reaches the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"\b(ckda_\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    from gated_delta_rule_ckda_gb300 import build
    build.build()
    import gated_delta_rule_ckda_gb300 as ck
    return ck.lib()


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "ckda_fwd" in names and "ckda_decode_step" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_status_strings_and_version(L):
    assert L.ckda_version() == 10000
    for code, name in [(0, b"CKDA_OK"), (1, b"CKDA_ERR_INVALID_ARG"), (4, b"CKDA_ERR_TIMEOUT"),
                       (6, b"CKDA_ERR_RANGE")]:
        assert L.ckda_status_string(code) == name
    assert L.ckda_status_string(99) == b"CKDA_ERR_UNKNOWN"


def test_workspace_bytes(L):
    assert L.ckda_fwd_workspace_bytes(0, 16) == 256
    assert L.ckda_fwd_workspace_bytes(64, 16) == 512
    assert L.ckda_fwd_workspace_bytes(65, 16) == 768


def _fwd(L, **kw):
    a = dict(q=1, k=1, v=1, alpha=1, beta=1, h0=None, o=1, hT=None, cu=None, num_seqs=0,
             B=1, H=1, T=4, dk=128, dv=128, io=1, scale=1.0, chunk=0, ws=None, wsb=0,
             stream=None)
    a.update(kw)
    vp = ctypes.c_void_p
    return L.ckda_fwd(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["alpha"]), vp(a["beta"]),
                      vp(a["h0"]), vp(a["o"]), vp(a["hT"]), vp(a["cu"]), a["num_seqs"], a["B"],
                      a["H"], a["T"], a["dk"], a["dv"], a["io"], a["scale"], a["chunk"],
                      vp(a["ws"]), a["wsb"], vp(a["stream"]))


def test_fwd_argument_errors_are_synchronous(L):
    INV, UNS, WS = 1, 2, 5
    assert _fwd(L, q=None) == INV
    assert _fwd(L, o=None) == INV
    assert _fwd(L, B=0) == INV
    assert _fwd(L, H=0) == INV
    assert _fwd(L, T=-1) == INV
    assert _fwd(L, io=7) == INV
    assert _fwd(L, scale=float("nan")) == INV
    assert _fwd(L, cu=16, num_seqs=2, B=2) == INV        # packed needs B == 1
    assert _fwd(L, cu=16, num_seqs=0) == INV             # packed needs >= 1 sequence
    assert _fwd(L, num_seqs=3, B=2) == INV
    assert _fwd(L, dk=129) == UNS
    assert _fwd(L, dv=256) == UNS
    assert _fwd(L, chunk=48) == UNS
    assert _fwd(L, chunk=16) == UNS                       # tensor-core path is chunk 64
    assert _fwd(L, ws=None) == WS
    assert _fwd(L, ws=4096, wsb=16) == WS                 # too small
    assert _fwd(L, ws=4096 + 8, wsb=4096) == WS          # misaligned
    assert _fwd(L, q=8, ws=4096, wsb=4096) == INV         # TMA base not 16-byte aligned


def test_decode_argument_errors_are_synchronous(L):
    vp = ctypes.c_void_p
    f = lambda **kw: L.ckda_decode_step(*(vp(kw.get(n, 1)) for n in
                                          ("q", "k", "v", "alpha", "beta", "state", "o")),
                                        kw.get("B", 1), kw.get("H", 1), kw.get("dk", 128),
                                        kw.get("dv", 128), kw.get("io", 1), 1.0, vp(None))
    assert f(state=None) == 1
    assert f(B=0) == 1
    assert f(dk=200) == 2
    assert f(state=4) == 1  # misaligned state for the vectorised kernel
    assert f(io=3) == 1


def test_decode_raw_argument_errors_are_synchronous(L):
    vp = ctypes.c_void_p
    names = ("q", "k", "v", "a", "b", "state", "o")
    f = lambda **kw: L.ckda_decode_step_raw(*(vp(kw.get(n, 256)) for n in names),
                                            kw.get("B", 1), kw.get("H", 1), kw.get("dk", 128),
                                            kw.get("dv", 128), kw.get("io", 1),
                                            ctypes.c_float(1.0), 1,
                                            ctypes.c_float(kw.get("eps", 1e-6)), vp(None))
    assert f(state=None) == 1
    assert f(b=None) == 1
    assert f(B=0) == 1
    assert f(dk=64) == 2          # the fused step is 128 x 128 only
    assert f(state=8) == 1        # misaligned state
    assert f(io=3) == 1
    assert f(eps=-1.0) == 1


def test_bwd_argument_errors_are_synchronous(L):
    vp = ctypes.c_void_p
    names = ("q", "k", "v", "alpha", "beta", "h0", "do", "dhT", "dq", "dk", "dv", "dalpha",
             "dbeta", "dh0", "cu")

    def f(**kw):
        ptrs = [vp(kw.get(n, 256 if n not in ("h0", "dhT", "dh0", "cu") else None))
                for n in names]
        return L.ckda_bwd(*ptrs, kw.get("nseq", 0), kw.get("B", 1), kw.get("H", 1),
                          kw.get("T", 4), kw.get("dk", 16), kw.get("dv", 16), kw.get("io", 0),
                          ctypes.c_float(1.0), vp(kw.get("ws", 256)),
                          ctypes.c_size_t(kw.get("wsb", 1 << 20)), vp(None))
    assert f(q=None) == 1
    assert f(dalpha=None) == 1
    assert f(B=0) == 1
    assert f(dk=129) == 2
    assert f(io=3) == 1
    assert f(cu=256, B=2, nseq=2) == 1      # packed input needs B == 1
    assert f(wsb=100) == 5                   # workspace smaller than needed
    assert f(ws=8) == 5                      # misaligned workspace
    # one state slice is one CTA's 32 columns: 256 threads x 16 rows of fp32; a
    # (sequence, head) has ceil(dv / 32) CTAs, each with 32 sub-checkpoint
    # slices (one per 2 tokens of a 64-token chunk)
    sl = 256 * 16 * 4
    # dense: ceil(T/64) checkpoints per (batch, head)
    assert L.ckda_bwd_workspace_bytes(0, 2, 3, 130, 16, 8) == (2 * 3 * 3 + 2 * 3 * 32) * sl
    assert L.ckda_bwd_workspace_bytes(0, 2, 3, 130, 16, 40) == 2 * (2 * 3 * 3 + 2 * 3 * 32) * sl
    # packed: ceil(T/64) + num_seqs checkpoints per head
    assert L.ckda_bwd_workspace_bytes(5, 1, 3, 130, 16, 8) == (3 * (3 + 5) + 5 * 3 * 32) * sl


def test_prep_argument_errors_are_synchronous(L):
    vp = ctypes.c_void_p
    names = ("q_raw", "k_raw", "a_raw", "b_raw", "q", "k", "alpha", "beta")
    f = lambda **kw: L.ckda_prep(*(vp(kw.get(n, 16)) for n in names), kw.get("rows", 4),
                                 kw.get("dk", 128), kw.get("io", 1), 1,
                                 ctypes.c_float(kw.get("eps", 1e-6)), vp(None))
    assert f(k_raw=None) == 1
    assert f(beta=None) == 1
    assert f(q=None) == 1          # q_raw given without q
    assert f(rows=-1) == 1
    assert f(dk=0) == 1
    assert f(dk=129) == 2
    assert f(io=3) == 1
    assert f(eps=-1.0) == 1
    assert f(eps=float("nan")) == 1
    # no rows: nothing to do, nothing launched
    assert f(rows=0, k_raw=None, beta=None) == 0


def test_prep_bwd_argument_errors_are_synchronous(L):
    vp = ctypes.c_void_p
    names = ("q_raw", "k_raw", "a_raw", "b_raw", "d_q", "d_k", "d_alpha", "d_beta", "d_q_raw",
             "d_k_raw", "d_a_raw", "d_b_raw")
    L.ckda_prep_bwd.argtypes = [vp] * 12 + [ctypes.c_longlong, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_float, vp]
    f = lambda **kw: L.ckda_prep_bwd(*(vp(kw.get(n, 16)) for n in names), kw.get("rows", 4),
                                     kw.get("dk", 128), kw.get("io", 1), 1,
                                     ctypes.c_float(kw.get("eps", 1e-6)), vp(None))
    assert f(k_raw=None) == 1
    assert f(d_beta=None) == 1
    assert f(d_a_raw=None) == 1
    assert f(d_q=None) == 1          # q_raw given without d_q
    assert f(d_q_raw=None) == 1      # ... or without d_q_raw
    assert f(rows=-1) == 1
    assert f(dk=0) == 1
    assert f(dk=129) == 2
    assert f(io=3) == 1
    assert f(eps=-1.0) == 1
    assert f(eps=float("nan")) == 1
    # no rows: nothing to do, nothing launched
    assert f(rows=0, k_raw=None, d_b_raw=None) == 0
    # no query at all is valid (and with no rows launches nothing)
    assert f(rows=0, q_raw=None, d_q=None, d_q_raw=None) == 0


def test_fwd_host_argument_errors_are_synchronous(L):
    """ckda_fwd_host rejects bad arguments, slices and scratch before any copy."""
    vp = ctypes.c_void_p
    B, H, T, d = 2, 3, 200, 128
    need = L.ckda_fwd_host_scratch_bytes(B, H, T, d, d, 1, 64)

    def f(**kw):
        return L.ckda_fwd_host(*(vp(kw.get(n, 16)) for n in ("q", "k", "v", "alpha", "beta")),
                               vp(kw.get("h0")), vp(kw.get("o", 16)), vp(kw.get("hT")),
                               kw.get("B", B), kw.get("H", H), kw.get("T", T), kw.get("dk", d),
                               kw.get("dv", d), kw.get("io", 1), kw.get("scale", 1.0),
                               kw.get("slice", 64), vp(kw.get("ws", 4096)),
                               kw.get("wsb", need), vp(None))
    assert f(q=None) == 1
    assert f(o=None) == 1
    assert f(B=0) == 1
    assert f(io=5) == 1
    assert f(slice=100) == 1                              # not a multiple of 64
    assert f(slice=-64) == 1
    assert f(scale=float("nan")) == 1
    assert f(dk=130) == 2
    assert f(ws=None) == 5
    assert f(wsb=need - 1) == 5                           # too small
    assert f(ws=4096 + 16) == 5                           # misaligned


def test_fwd_host_scratch_bytes(L):
    """Two slice buffers (q, k, alpha, v, beta, o) plus the carried state and
    the status word; the automatic slice is about T / 4, at least 512."""
    f = L.ckda_fwd_host_scratch_bytes
    B, H, d = 2, 3, 128
    up = lambda x: (x + 255) // 256 * 256
    for T, sl, ts in ((1000, 64, 64), (1000, 128, 128), (2048, 0, 512), (8192, 0, 2048),
                      (1000, 0, 512), (100, 0, 128)):
        rows = B * H * ts
        buf = 4 * up(rows * d * 2) + up(rows * 2) + up(rows * d * 2)
        assert f(B, H, T, d, d, 1, sl) == 256 + up(B * H * d * d * 4) + 2 * buf, (T, sl)
    assert f(B, H, 1000, d, d, 1, 100) == 0
    assert f(0, H, 1000, d, d, 1, 64) == 0


def test_selftest_rejects_missing_workspace(L):
    assert L.ckda_selftest_timeout(None, 0, 10, None) == 5


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import gated_delta_rule_ckda_gb300 as ck
    monkeypatch.setattr(ck, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ck, "_lib", None)
    with pytest.raises(ImportError):
        ck.lib()


def _split_model(B, H, T, sms):
    """The segment-count rule ckda_fwd_split_segments documents, restated:
    both passes in whole waves of CTAs, plus 2 + (S - 2) / 2 chunk steps, and a
    count must beat one plain pass by 10%."""
    units, nch = B * H, (T + 63) // 64
    waves = lambda n: -(-n // sms)
    best, best_s = waves(units) * nch, 1
    for S in range(2, min(16, nch) + 1):
        sc = -(-nch // S)
        if -(-nch // sc) != S:
            continue
        p1 = 2 * S - 3 if S >= 3 else 1
        t = (waves(units * p1) + waves(units * (S - 1))) * sc + 2.0 + 0.5 * (S - 2)
        if t < 0.9 * best:
            best, best_s = t, S
    return best_s


def test_split_segments_rule(L):
    f = L.ckda_fwd_split_segments
    assert f(1, 16, 32768, 128, 128, 0, 152) == 1       # fp32: not the tensor-core path
    assert f(1, 16, 32768, 96, 128, 1, 152) == 1        # dk 96: not the tensor-core path
    assert f(8, 16, 2048, 128, 128, 1, 152) == 1        # 128 units already fill the GPU
    assert f(1, 16, 64, 128, 128, 1, 152) == 1          # one chunk
    assert f(0, 16, 32768, 128, 128, 1, 152) == 1       # bad size
    for B, H, T, dk in ((1, 16, 32768, 128), (1, 1, 5000, 128), (2, 8, 20000, 64),
                        (1, 32, 8192, 128), (1, 4, 700, 128)):
        assert f(B, H, T, dk, 128, 1, 152) == _split_model(B, H, T, 152), (B, H, T)
    s = f(1, 16, 32768, 128, 128, 1, 152)
    assert s >= 6 and 16 * (2 * s - 3) <= 2 * 152


def test_split_workspace_bytes(L):
    f = L.ckda_fwd_split_workspace_bytes
    tile = 128 * 128 * 4
    assert f(1, 2, 1000, 128, 128, 1, 1) == 256
    assert f(1, 2, 1000, 128, 128, 1, 2) == 256 + 1 * 2 * 2 * tile       # 16 chunks: 2 x 8
    assert f(1, 2, 1000, 128, 128, 1, 4) == 256 + 3 * 2 * 4 * tile       # 4 x 4
    assert f(1, 2, 1000, 128, 128, 1, 5) == 256 + 3 * 2 * 4 * tile       # 4 chunks each: 4
    assert f(1, 2, 1000, 64, 128, 1, 4) == 256 + 3 * 2 * 4 * tile // 2
    assert f(2, 3, 100, 128, 128, 1, 16) == 256 + 1 * 6 * 2 * tile       # 2 chunks: 2 segments
    assert f(1, 2, 0, 128, 128, 1, 4) == 256
    assert f(1, 2, 1000, 128, 128, 1, -1) == 0


def test_split_argument_errors_are_synchronous(L):
    """ckda_fwd_split rejects bad arguments and workspaces before launching."""
    vp = ctypes.c_void_p
    B, H, T, d = 1, 2, 1000, 128
    need = L.ckda_fwd_split_workspace_bytes(B, H, T, d, d, 1, 4)

    def f(**kw):
        return L.ckda_fwd_split(*(vp(kw.get(n, 16)) for n in ("q", "k", "v", "alpha", "beta")),
                                vp(kw.get("h0")), vp(kw.get("o", 16)), vp(kw.get("hT")),
                                kw.get("B", B), kw.get("H", H), kw.get("T", T), kw.get("dk", d),
                                kw.get("dv", d), kw.get("io", 1), kw.get("scale", 1.0),
                                kw.get("seg", 4), vp(kw.get("ws", 4096)), kw.get("wsb", need),
                                vp(None))
    assert f(seg=-1) == 1
    assert f(q=None) == 1
    assert f(o=None) == 1
    assert f(B=0) == 1
    assert f(io=5) == 1
    assert f(scale=float("nan")) == 1
    assert f(q=16 + 2) == 1                               # TMA bases must be 16-byte aligned
    assert f(io=0) == 2                                   # fp32: no split path
    assert f(dk=96) == 2
    assert f(dv=64) == 2
    assert f(ws=None) == 5
    assert f(wsb=need - 1) == 5
    assert f(ws=4096 + 16) == 5


def test_split_varlen_workspace_and_segment_length(L):
    """Workspace: status word and order (rounded to 256 B), the plan (4 N + 3
    int32, rounded to 256 B), then three state tiles per segment slot, with
    T // seg_len + 1 + N slots (an upper bound on sum_i max(1, ceil(L_i /
    seg_len)) for any lengths summing to T)."""
    f = L.ckda_fwd_split_varlen_workspace_bytes
    tile = 128 * 128 * 4
    r256 = lambda x: (x + 255) // 256 * 256
    for N, H, T, dk, sl in ((4, 2, 1000, 128, 256), (64, 16, 528000, 128, 4096),
                            (1, 1, 0, 64, 64), (3, 5, 777, 64, 192)):
        slots = T // sl + 1 + N
        want = r256(256 + 4 * N) + r256(4 * (4 * N + 3)) + 3 * slots * H * tile * dk // 128
        assert f(N, H, T, dk, sl) == want, (N, H, T, dk, sl)
    assert f(4, 2, 1000, 128, 100) == 0      # not a multiple of 64
    assert f(4, 2, 1000, 128, 0) == 0
    assert f(0, 2, 1000, 128, 256) == 0
    # automatic segment length: the average work per SM in chunk steps (at
    # least 16 chunks), 0 off the tensor-core path
    g = L.ckda_fwd_split_varlen_seg_len
    for N, H, T in ((64, 16, 528000), (64, 16, 97280), (1, 1, 64), (8, 4, 100000)):
        work = ((T + 63) // 64 + N) * H
        assert g(N, H, T, 128, 128, 1, 152) == max(16, -(-work // 152)) * 64, (N, H, T)
    assert g(4, 2, 1000, 128, 128, 0, 152) == 0     # fp32
    assert g(4, 2, 1000, 96, 128, 1, 152) == 0      # dk 96
    assert g(0, 2, 1000, 128, 128, 1, 152) == 0


def test_split_varlen_argument_errors_are_synchronous(L):
    vp = ctypes.c_void_p
    N, H, T, d = 3, 2, 1000, 128
    need = L.ckda_fwd_split_varlen_workspace_bytes(N, H, T, d, 256)

    def f(**kw):
        return L.ckda_fwd_split_varlen(
            *(vp(kw.get(n, 16)) for n in ("q", "k", "v", "alpha", "beta")), vp(kw.get("h0")),
            vp(kw.get("o", 16)), vp(kw.get("hT")), vp(kw.get("cu", 16)), kw.get("N", N),
            kw.get("H", H), kw.get("T", T), kw.get("dk", d), kw.get("dv", d), kw.get("io", 1),
            kw.get("scale", 1.0), kw.get("seg", 256), vp(kw.get("ws", 4096)), kw.get("wsb", need),
            vp(None))
    assert f(cu=None) == 1
    assert f(N=0) == 1
    assert f(seg=100) == 1                     # not a multiple of 64
    assert f(seg=-64) == 1
    assert f(q=None) == 1
    assert f(q=16 + 2) == 1                    # TMA bases must be 16-byte aligned
    assert f(scale=float("nan")) == 1
    assert f(io=0) == 2                        # fp32: no tensor-core path
    assert f(dk=96) == 2
    assert f(ws=None) == 5
    assert f(wsb=need - 1) == 5
    assert f(ws=4096 + 16) == 5


def test_fwd_raw_argument_errors_are_synchronous(L):
    """ckda_fwd_raw takes ckda_fwd's checks, the tensor-core shapes only, and a
    valid norm_eps."""
    vp = ctypes.c_void_p
    B, H, T, d = 2, 3, 100, 128
    need = L.ckda_fwd_workspace_bytes(0, H)

    def f(**kw):
        return L.ckda_fwd_raw(*(vp(kw.get(n, 16)) for n in ("q", "k", "v", "a", "b")),
                              vp(kw.get("h0")), vp(kw.get("o", 16)), vp(kw.get("hT")),
                              vp(kw.get("cu")), kw.get("N", 0), kw.get("B", B), kw.get("H", H),
                              kw.get("T", T), kw.get("dk", d), kw.get("dv", d), kw.get("io", 1),
                              kw.get("scale", 1.0), kw.get("nq", 1), kw.get("eps", 1e-6),
                              vp(kw.get("ws", 4096)), kw.get("wsb", need), vp(None))
    assert f(q=None) == 1
    assert f(B=0) == 1
    assert f(eps=-1.0) == 1
    assert f(eps=float("nan")) == 1
    assert f(io=0) == 2          # fp32: ckda_prep then ckda_fwd
    assert f(dk=96) == 2
    assert f(dv=64) == 2
    assert f(q=16 + 2) == 1      # TMA bases must be 16-byte aligned
    assert f(ws=None) == 5
