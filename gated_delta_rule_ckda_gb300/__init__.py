"""Python binding of libckda -- the GB300 (sm_103a) Complex KDA recurrence.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libckda.so (csrc/), called through its C ABI (include/ckda.h).
PyTorch supplies device memory and streams.  There is no CPU or PyTorch
fallback: if the library is missing or fails to load, every call raises.

    o, hT = fwd(q, k, v, alpha, beta, h0=None, cu_seqlens=None, scale=1.0)
    o = decode_step(q, k, v, alpha, beta, state)      # state updated in place

Shapes follow the C ABI: q, k, alpha [B, H, T, dk]; v [B, H, T, dv];
beta [B, H, T]; h0 / hT fp32 [N, H, dk, dv] with N = B, or the number of
packed sequences when cu_seqlens (int32 [N + 1], B == 1) is given.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["fwd", "fwd_host", "fwd_split", "decode_step", "decode_step_raw", "prep", "bwd",
           "bwd_workspace_bytes", "fwd_status", "workspace_bytes", "split_segments",
           "split_workspace_bytes", "host_scratch_bytes", "selftest_timeout", "lib",
           "library_path", "CkdaError", "STATUS", "recurrence", "prepare"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libckda.so")
_lock = threading.Lock()
_lib = None

STATUS = {0: "CKDA_OK", 1: "CKDA_ERR_INVALID_ARG", 2: "CKDA_ERR_UNSUPPORTED",
          3: "CKDA_ERR_CUDA", 4: "CKDA_ERR_TIMEOUT", 5: "CKDA_ERR_WORKSPACE",
          6: "CKDA_ERR_RANGE"}
_F32, _BF16 = 0, 1


class CkdaError(RuntimeError):
    def __init__(self, code, where):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS.get(self.code, self.code)}")


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libckda (ctypes.CDLL).  Raises if the library is not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(
                    f"libckda.so is not built ({_LIB_PATH}); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(_LIB_PATH)
            vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
            L.ckda_version.restype = i32
            L.ckda_version.argtypes = []
            L.ckda_status_string.restype = ctypes.c_char_p
            L.ckda_status_string.argtypes = [i32]
            L.ckda_fwd_workspace_bytes.restype = sz
            L.ckda_fwd_workspace_bytes.argtypes = [i32, i32]
            L.ckda_fwd.restype = i32
            L.ckda_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                   i32, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
            L.ckda_fwd_status.restype = i32
            L.ckda_fwd_status.argtypes = [vp, vp]
            L.ckda_decode_step.restype = i32
            L.ckda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp,
                                           i32, i32, i32, i32, i32, f32, vp]
            L.ckda_selftest_timeout.restype = i32
            L.ckda_selftest_timeout.argtypes = [vp, sz, ctypes.c_uint, vp]
            L.ckda_fwd_host_scratch_bytes.restype = sz
            L.ckda_fwd_host_scratch_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
            L.ckda_decode_step_raw.restype = i32
            L.ckda_decode_step_raw.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                               i32, f32, i32, f32, vp]
            L.ckda_bwd_workspace_bytes.restype = sz
            L.ckda_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
            L.ckda_bwd.restype = i32
            L.ckda_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                   i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp]
            L.ckda_prep.restype = i32
            L.ckda_prep.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_longlong, i32, i32,
                                    i32, f32, vp]
            L.ckda_fwd_split_varlen_seg_len.restype = i32
            L.ckda_fwd_split_varlen_seg_len.argtypes = [i32] * 7
            L.ckda_fwd_split_varlen_workspace_bytes.restype = sz
            L.ckda_fwd_split_varlen_workspace_bytes.argtypes = [i32] * 5
            L.ckda_fwd_split_varlen.restype = i32
            L.ckda_fwd_split_varlen.argtypes = [vp] * 9 + [i32] * 6 + [f32, i32, vp, sz, vp]
            L.ckda_fwd_raw.restype = i32
            L.ckda_fwd_raw.argtypes = [vp] * 9 + [i32] * 7 + [f32, i32, f32, vp, sz, vp]
            L.ckda_prep_bwd.restype = i32
            L.ckda_prep_bwd.argtypes = [vp] * 12 + [ctypes.c_longlong, i32, i32, i32, f32, vp]
            L.ckda_fwd_host.restype = i32
            L.ckda_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                        i32, f32, i32, vp, sz, vp]
            L.ckda_fwd_split_segments.restype = i32
            L.ckda_fwd_split_segments.argtypes = [i32, i32, i32, i32, i32, i32, i32]
            L.ckda_fwd_split_workspace_bytes.restype = sz
            L.ckda_fwd_split_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
            L.ckda_fwd_split.restype = i32
            L.ckda_fwd_split.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                         i32, f32, i32, vp, sz, vp]
            _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _io_dtype(t):
    if t.dtype == torch.bfloat16:
        return _BF16
    if t.dtype == torch.float32:
        return _F32
    raise TypeError(f"unsupported I/O dtype {t.dtype} (bf16 or fp32)")


def _check(t, name, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


def workspace_bytes(num_seqs: int, H: int) -> int:
    return int(lib().ckda_fwd_workspace_bytes(int(num_seqs), int(H)))


def new_workspace(num_seqs, H, device):
    n = workspace_bytes(num_seqs, H)
    return torch.empty(n, dtype=torch.uint8, device=device)


def fwd_raw(q_raw, k_raw, v, a_raw, b_raw, h0=None, cu_seqlens=None, scale=1.0,
            normalize_q=True, norm_eps=1e-6, store_final_state=True, o=None, hT=None,
            workspace=None, stream=None):
    """ckda_fwd_raw: the forward on raw q, k and gate logits a, b, with the
    input preparation of `prep` applied inside the kernel.  Returns (o, hT or
    None)."""
    return fwd(q_raw, k_raw, v, a_raw, b_raw, h0, cu_seqlens, scale, 0, store_final_state, o,
               hT, workspace, stream, _raw=(bool(normalize_q), float(norm_eps)))


def fwd(q, k, v, alpha, beta, h0=None, cu_seqlens=None, scale=1.0, chunk_size=0,
        store_final_state=True, o=None, hT=None, workspace=None, stream=None, _raw=None):
    """Forward over [B, H, T, d] (or packed) inputs.  Returns (o, hT or None)."""
    L = lib()
    device = q.device
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    _io_dtype(q)
    for name, t, shp in (("q", q, (B, H, T, dk)), ("k", k, (B, H, T, dk)),
                         ("alpha", alpha, (B, H, T, dk)), ("v", v, (B, H, T, dv)),
                         ("beta", beta, (B, H, T))):
        _check(t, name, dt, shp, device)
    N = B
    if cu_seqlens is not None:
        N = cu_seqlens.numel() - 1
        _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), device)
    if h0 is not None:
        _check(h0, "h0", torch.float32, (N, H, dk, dv), device)
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=dt, device=device)
    else:
        _check(o, "o", dt, (B, H, T, dv), device)
    if store_final_state and hT is None:
        hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=device)
    if hT is not None:
        _check(hT, "hT", torch.float32, (N, H, dk, dv), device)
    nseq_ws = N if cu_seqlens is not None else 0
    if workspace is None:
        workspace = new_workspace(nseq_ws, H, device)
    nseq = int(N if cu_seqlens is not None else 0)
    if _raw is None:
        rc = L.ckda_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(h0), _ptr(o),
                        _ptr(hT), _ptr(cu_seqlens), nseq, B, H, T, dk, dv, _io_dtype(q),
                        float(scale), int(chunk_size), _ptr(workspace), int(workspace.numel()),
                        _stream_handle(stream, device))
    else:
        rc = L.ckda_fwd_raw(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(h0), _ptr(o),
                            _ptr(hT), _ptr(cu_seqlens), nseq, B, H, T, dk, dv, _io_dtype(q),
                            float(scale), int(_raw[0]), float(_raw[1]), _ptr(workspace),
                            int(workspace.numel()), _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_fwd" if _raw is None else "ckda_fwd_raw")
    fwd.last_workspace = workspace
    fwd_raw.last_workspace = workspace
    return o, hT


def split_segments(B, H, T, dk, dv, dtype=torch.bfloat16, num_sms=0) -> int:
    """Segment count ckda_fwd_split picks for `segments=0` (num_sms = 0: the
    current device's SM count)."""
    io = _BF16 if dtype == torch.bfloat16 else _F32
    return int(lib().ckda_fwd_split_segments(B, H, T, dk, dv, io, int(num_sms)))


def split_workspace_bytes(B, H, T, dk, dv, dtype=torch.bfloat16, segments=0) -> int:
    io = _BF16 if dtype == torch.bfloat16 else _F32
    return int(lib().ckda_fwd_split_workspace_bytes(B, H, T, dk, dv, io, int(segments)))


def fwd_split(q, k, v, alpha, beta, h0=None, scale=1.0, segments=0, store_final_state=True,
              o=None, hT=None, workspace=None, stream=None):
    """ckda_fwd_split: the dense forward with each sequence cut into segments
    run in parallel (two passes and a scan of the segment operators).
    Returns (o, hT or None)."""
    L = lib()
    device = q.device
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    io = _io_dtype(q)
    for name, t, shp in (("q", q, (B, H, T, dk)), ("k", k, (B, H, T, dk)),
                         ("alpha", alpha, (B, H, T, dk)), ("v", v, (B, H, T, dv)),
                         ("beta", beta, (B, H, T))):
        _check(t, name, dt, shp, device)
    if h0 is not None:
        _check(h0, "h0", torch.float32, (B, H, dk, dv), device)
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=dt, device=device)
    else:
        _check(o, "o", dt, (B, H, T, dv), device)
    if store_final_state and hT is None:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=device)
    if hT is not None:
        _check(hT, "hT", torch.float32, (B, H, dk, dv), device)
    if workspace is None:
        with torch.cuda.device(device):
            n = int(L.ckda_fwd_split_workspace_bytes(B, H, T, dk, dv, io, int(segments)))
        workspace = torch.empty(n, dtype=torch.uint8, device=device)
    with torch.cuda.device(device):
        rc = L.ckda_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(h0),
                              _ptr(o), _ptr(hT), B, H, T, dk, dv, io, float(scale),
                              int(segments), _ptr(workspace), int(workspace.numel()),
                              _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_fwd_split")
    fwd_split.last_workspace = workspace
    return o, hT


def split_varlen_seg_len(num_seqs, H, T, dk, dv, dtype=torch.bfloat16, num_sms=0) -> int:
    """Segment length ckda_fwd_split_varlen picks for `seg_len=0`."""
    io = _BF16 if dtype == torch.bfloat16 else _F32
    return int(lib().ckda_fwd_split_varlen_seg_len(num_seqs, H, T, dk, dv, io, int(num_sms)))


def split_varlen_workspace_bytes(num_seqs, H, T, dk, seg_len) -> int:
    return int(lib().ckda_fwd_split_varlen_workspace_bytes(num_seqs, H, T, dk, int(seg_len)))


def fwd_split_varlen(q, k, v, alpha, beta, cu_seqlens, h0=None, scale=1.0, seg_len=0,
                     store_final_state=True, o=None, hT=None, workspace=None, stream=None):
    """ckda_fwd_split_varlen: the packed forward with every sequence longer
    than seg_len cut into segments run in parallel.  q, k, alpha, v are
    [1, H, T, d], beta [1, H, T], cu_seqlens int32 [N + 1] on the device.
    Returns (o, hT [N, H, dk, dv] or None)."""
    L = lib()
    device = q.device
    B, H, T, dk = q.shape
    if B != 1:
        raise ValueError("fwd_split_varlen: packed input has B = 1")
    dv = v.shape[-1]
    dt = q.dtype
    io = _io_dtype(q)
    for name, t, shp in (("q", q, (1, H, T, dk)), ("k", k, (1, H, T, dk)),
                         ("alpha", alpha, (1, H, T, dk)), ("v", v, (1, H, T, dv)),
                         ("beta", beta, (1, H, T))):
        _check(t, name, dt, shp, device)
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.device != device or cu_seqlens.dim() != 1:
        raise ValueError("fwd_split_varlen: cu_seqlens must be int32 [N + 1] on the device")
    N = cu_seqlens.numel() - 1
    if h0 is not None:
        _check(h0, "h0", torch.float32, (N, H, dk, dv), device)
    if o is None:
        o = torch.empty((1, H, T, dv), dtype=dt, device=device)
    else:
        _check(o, "o", dt, (1, H, T, dv), device)
    if store_final_state and hT is None:
        hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=device)
    if hT is not None:
        _check(hT, "hT", torch.float32, (N, H, dk, dv), device)
    with torch.cuda.device(device):
        if seg_len == 0:
            seg_len = int(L.ckda_fwd_split_varlen_seg_len(N, H, T, dk, dv, io, 0))
        if workspace is None:
            n = int(L.ckda_fwd_split_varlen_workspace_bytes(N, H, T, dk, int(seg_len)))
            workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        rc = L.ckda_fwd_split_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(h0),
                                     _ptr(o), _ptr(hT), _ptr(cu_seqlens), N, H, T, dk, dv, io,
                                     float(scale), int(seg_len), _ptr(workspace),
                                     int(workspace.numel()), _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_fwd_split_varlen")
    fwd_split_varlen.last_workspace = workspace
    return o, hT


def fwd_status(workspace, stream=None) -> int:
    """Device status of the most recent call on `workspace` (synchronises)."""
    return int(lib().ckda_fwd_status(_ptr(workspace), _stream_handle(stream, workspace.device)))


def host_scratch_bytes(B, H, T, dk, dv, dtype=torch.bfloat16, slice_tokens=0) -> int:
    io = _BF16 if dtype == torch.bfloat16 else _F32
    return int(lib().ckda_fwd_host_scratch_bytes(B, H, T, dk, dv, io, int(slice_tokens)))


def fwd_host(q, k, v, alpha, beta, h0=None, scale=1.0, slice_tokens=0, o=None, hT=None,
             store_final_state=True, scratch=None, stream=None, device=None):
    """ckda_fwd_host: the dense forward with every tensor in host memory (CPU
    tensors; pinned memory copies at full speed).  The copies of one slice of
    tokens overlap the computation of another.  Returns (o, hT or None) as CPU
    tensors; they are complete once `stream` is (this call does not wait)."""
    L = lib()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    io = _io_dtype(q)
    cpu = torch.device("cpu")
    for name, t, shp in (("q", q, (B, H, T, dk)), ("k", k, (B, H, T, dk)),
                         ("alpha", alpha, (B, H, T, dk)), ("v", v, (B, H, T, dv)),
                         ("beta", beta, (B, H, T))):
        _check(t, name, dt, shp, cpu)
    if h0 is not None:
        _check(h0, "h0", torch.float32, (B, H, dk, dv), cpu)
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=dt).pin_memory()
    else:
        _check(o, "o", dt, (B, H, T, dv), cpu)
    if store_final_state and hT is None:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32).pin_memory()
    if hT is not None:
        _check(hT, "hT", torch.float32, (B, H, dk, dv), cpu)
    need = host_scratch_bytes(B, H, T, dk, dv, dt, slice_tokens)
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=device)
    rc = L.ckda_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(h0), _ptr(o),
                         _ptr(hT), B, H, T, dk, dv, io, float(scale), int(slice_tokens),
                         _ptr(scratch), int(scratch.numel()), _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_fwd_host")
    fwd_host.last_scratch = scratch
    return o, hT


def decode_step(q, k, v, alpha, beta, state, scale=1.0, o=None, stream=None):
    """One token per (batch, head); `state` [B, H, dk, dv] fp32 is updated in place."""
    L = lib()
    device = q.device
    B, H, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    _io_dtype(q)
    for name, t, shp in (("q", q, (B, H, dk)), ("k", k, (B, H, dk)), ("alpha", alpha, (B, H, dk)),
                         ("v", v, (B, H, dv)), ("beta", beta, (B, H))):
        _check(t, name, dt, shp, device)
    _check(state, "state", torch.float32, (B, H, dk, dv), device)
    if o is None:
        o = torch.empty((B, H, dv), dtype=dt, device=device)
    else:
        _check(o, "o", dt, (B, H, dv), device)
    rc = L.ckda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(state),
                            _ptr(o), B, H, dk, dv, _io_dtype(q), float(scale),
                            _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_decode_step")
    return o


def selftest_timeout(workspace, spin_limit=1000, stream=None) -> int:
    """Runs the bounded-wait self-test and returns the status it recorded."""
    L = lib()
    rc = L.ckda_selftest_timeout(_ptr(workspace), int(workspace.numel()), int(spin_limit),
                                 _stream_handle(stream, workspace.device))
    if rc != 0:
        raise CkdaError(rc, "ckda_selftest_timeout")
    return fwd_status(workspace, stream)


def fwd_noalloc(q, k, v, alpha, beta, h0=None, cu_seqlens=None, scale=1.0, chunk_size=0,
                o=None, hT=None, stream=None):
    """ckda_fwd_noalloc: the forward without a workspace, for callers that may
    not allocate device memory (its scratch is a fixed array inside libckda).
    o and hT may be passed in so that the call itself allocates nothing."""
    L = lib()
    fn = L.ckda_fwd_noalloc
    if fn.argtypes is None:
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                       i32, i32, i32, i32, i32, i32, f32, i32, vp]
        fn.restype = i32
    device = q.device
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=q.dtype, device=device)
    if hT is None:
        hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=device)
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(h0), _ptr(o), _ptr(hT),
            _ptr(cu_seqlens), int(N if cu_seqlens is not None else 0), B, H, T, dk, dv,
            _io_dtype(q), float(scale), int(chunk_size), _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_fwd_noalloc")
    return o, hT


def prep(k_raw, a_raw, b_raw, q_raw=None, normalize_q=True, norm_eps=1e-6, out=None,
         stream=None):
    """Fused input preparation (ckda_prep): unit-norm keys (and queries when
    normalize_q), alpha = s[e^-5 + (1 - e^-5)|tanh(a/2)|], beta = 2 sigmoid(b).

    k_raw, a_raw (and q_raw) are [..., dk]; b_raw is [...].  Returns
    (q or None, k, alpha, beta) in the input dtype.  `out` may give the four
    output tensors (q may be None); passing the inputs themselves works in place.
    """
    L = lib()
    device = k_raw.device
    dt = k_raw.dtype
    dk = k_raw.shape[-1]
    _check(a_raw, "a_raw", dt, tuple(k_raw.shape), device)
    _check(b_raw, "b_raw", dt, tuple(k_raw.shape[:-1]), device)
    if q_raw is not None:
        _check(q_raw, "q_raw", dt, tuple(k_raw.shape), device)
    _check(k_raw, "k_raw", dt, tuple(k_raw.shape), device)
    if out is None:
        q = None if q_raw is None else torch.empty_like(q_raw)
        k, alpha, beta = torch.empty_like(k_raw), torch.empty_like(a_raw), torch.empty_like(b_raw)
    else:
        q, k, alpha, beta = out
        for name, t, shp in (("k", k, k_raw.shape), ("alpha", alpha, k_raw.shape),
                             ("beta", beta, k_raw.shape[:-1])):
            _check(t, name, dt, tuple(shp), device)
        if (q is None) != (q_raw is None):
            raise ValueError("prep: q and q_raw must both be given or both be None")
        if q is not None:
            _check(q, "q", dt, tuple(k_raw.shape), device)
    rows = k_raw.numel() // dk if dk else 0
    rc = L.ckda_prep(_ptr(q_raw), _ptr(k_raw), _ptr(a_raw), _ptr(b_raw), _ptr(q), _ptr(k),
                     _ptr(alpha), _ptr(beta), int(rows), int(dk), _io_dtype(k_raw),
                     int(bool(normalize_q)), float(norm_eps), _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_prep")
    return q, k, alpha, beta


def prep_bwd(k_raw, a_raw, b_raw, d_k, d_alpha, d_beta, q_raw=None, d_q=None, normalize_q=True,
             norm_eps=1e-6, out=None, stream=None):
    """Backward of ``prep`` (ckda_prep_bwd): the gradients with respect to the
    raw inputs from those with respect to (q, k, alpha, beta).  The gate's
    sign carries no gradient and |tanh(a/2)| takes the subgradient 0 at a = 0.

    Returns (d_q_raw or None, d_k_raw, d_a_raw, d_b_raw) in the input dtype;
    `out` may give the four output tensors (d_q_raw may be None)."""
    L = lib()
    device = k_raw.device
    dt = k_raw.dtype
    shp = tuple(k_raw.shape)
    dk = shp[-1]
    for name, t, want in (("a_raw", a_raw, shp), ("b_raw", b_raw, shp[:-1]), ("d_k", d_k, shp),
                          ("d_alpha", d_alpha, shp), ("d_beta", d_beta, shp[:-1]),
                          ("k_raw", k_raw, shp)):
        _check(t, name, dt, want, device)
    if (q_raw is None) != (d_q is None):
        raise ValueError("prep_bwd: q_raw and d_q must both be given or both be None")
    if q_raw is not None:
        _check(q_raw, "q_raw", dt, shp, device)
        _check(d_q, "d_q", dt, shp, device)
    if out is None:
        dq_raw = None if q_raw is None else torch.empty_like(q_raw)
        dk_raw, da_raw, db_raw = (torch.empty_like(k_raw), torch.empty_like(a_raw),
                                  torch.empty_like(b_raw))
    else:
        dq_raw, dk_raw, da_raw, db_raw = out
        for name, t, want in (("d_k_raw", dk_raw, shp), ("d_a_raw", da_raw, shp),
                              ("d_b_raw", db_raw, shp[:-1])):
            _check(t, name, dt, want, device)
        if (dq_raw is None) != (q_raw is None):
            raise ValueError("prep_bwd: d_q_raw and q_raw must both be given or both be None")
        if dq_raw is not None:
            _check(dq_raw, "d_q_raw", dt, shp, device)
    rows = k_raw.numel() // dk if dk else 0
    rc = L.ckda_prep_bwd(_ptr(q_raw), _ptr(k_raw), _ptr(a_raw), _ptr(b_raw), _ptr(d_q),
                         _ptr(d_k), _ptr(d_alpha), _ptr(d_beta), _ptr(dq_raw), _ptr(dk_raw),
                         _ptr(da_raw), _ptr(db_raw), int(rows), int(dk), _io_dtype(k_raw),
                         int(bool(normalize_q)), float(norm_eps), _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_prep_bwd")
    return dq_raw, dk_raw, da_raw, db_raw


def bwd_workspace_bytes(B, H, T, dk, dv, num_seqs=0) -> int:
    return int(lib().ckda_bwd_workspace_bytes(num_seqs, B, H, T, dk, dv))


def bwd(q, k, v, alpha, beta, do, h0=None, dhT=None, cu_seqlens=None, scale=1.0,
        store_dh0=True, workspace=None, stream=None):
    """Backward of fwd (ckda_bwd): gradients of sum <o, do> + <hT, dhT>.

    Returns (dq, dk, dv, dalpha, dbeta, dh0 or None); dh0 is fp32."""
    L = lib()
    device = q.device
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    _io_dtype(q)
    for name, t, shp in (("q", q, (B, H, T, dk)), ("k", k, (B, H, T, dk)),
                         ("alpha", alpha, (B, H, T, dk)), ("v", v, (B, H, T, dv)),
                         ("do", do, (B, H, T, dv)), ("beta", beta, (B, H, T))):
        _check(t, name, dt, shp, device)
    N = B
    if cu_seqlens is not None:
        N = cu_seqlens.numel() - 1
        _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), device)
    for name, t in (("h0", h0), ("dhT", dhT)):
        if t is not None:
            _check(t, name, torch.float32, (N, H, dk, dv), device)
    need = bwd_workspace_bytes(B, H, T, dk, dv, N if cu_seqlens is not None else 0)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    dq, dkk, dal = torch.empty_like(q), torch.empty_like(k), torch.empty_like(alpha)
    dvv, dbe = torch.empty_like(v), torch.empty_like(beta)
    dh0 = torch.empty((N, H, dk, dv), dtype=torch.float32, device=device) if store_dh0 else None
    rc = L.ckda_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(h0), _ptr(do),
                    _ptr(dhT), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dal), _ptr(dbe), _ptr(dh0),
                    _ptr(cu_seqlens), int(N if cu_seqlens is not None else 0), B, H, T, dk, dv,
                    _io_dtype(q), float(scale), _ptr(workspace), int(workspace.numel()),
                    _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_bwd")
    return dq, dkk, dvv, dal, dbe, dh0


def decode_step_raw(q_raw, k_raw, v, a_raw, b_raw, state, scale=1.0, normalize_q=True,
                    norm_eps=1e-6, o=None, stream=None):
    """One decode step on raw inputs with the input preparation fused in
    (ckda_decode_step_raw): unit-norm k (and q), alpha and beta from the gate
    logits a and b.  state [B, H, 128, 128] fp32 is updated in place; returns o."""
    L = lib()
    device = q_raw.device
    B, H, dk = q_raw.shape
    dv = v.shape[-1]
    dt = q_raw.dtype
    for name, t, shp in (("q_raw", q_raw, (B, H, dk)), ("k_raw", k_raw, (B, H, dk)),
                         ("a_raw", a_raw, (B, H, dk)), ("v", v, (B, H, dv)),
                         ("b_raw", b_raw, (B, H))):
        _check(t, name, dt, shp, device)
    _check(state, "state", torch.float32, (B, H, dk, dv), device)
    if o is None:
        o = torch.empty((B, H, dv), dtype=dt, device=device)
    rc = L.ckda_decode_step_raw(_ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(a_raw), _ptr(b_raw),
                                _ptr(state), _ptr(o), B, H, dk, dv, _io_dtype(q_raw),
                                float(scale), int(bool(normalize_q)), float(norm_eps),
                                _stream_handle(stream, device))
    if rc != 0:
        raise CkdaError(rc, "ckda_decode_step_raw")
    return o


# ------------------------------------------------------------------- autograd
# Training use: the forward (fwd) with its backward (bwd), and the input
# preparation (prep) with its backward (prep_bwd), as torch.autograd
# functions.  They only route tensors between the calls above.

class _Recurrence(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, alpha, beta, h0, cu_seqlens, scale):
        o, hT = fwd(q, k, v, alpha, beta, h0, cu_seqlens, scale=scale)
        ctx.save_for_backward(q, k, v, alpha, beta, h0, cu_seqlens)
        ctx.scale = scale
        return o, hT

    @staticmethod
    def backward(ctx, do, dhT):
        q, k, v, alpha, beta, h0, cu = ctx.saved_tensors
        do = torch.zeros_like(v) if do is None else do.contiguous()
        dhT = None if dhT is None else dhT.contiguous()
        dq, dk, dv, da, db, dh0 = bwd(q, k, v, alpha, beta, do, h0=h0, dhT=dhT, cu_seqlens=cu,
                                      scale=ctx.scale, store_dh0=h0 is not None)
        return dq, dk, dv, da, db, dh0, None, None


def recurrence(q, k, v, alpha, beta, h0=None, cu_seqlens=None, scale=1.0):
    """(o, hT) = fwd(...), differentiable in q, k, v, alpha, beta and h0
    (the gradients come from bwd).  hT is fp32 [N, H, dk, dv]."""
    return _Recurrence.apply(q, k, v, alpha, beta, h0, cu_seqlens, float(scale))


class _Prepare(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q_raw, k_raw, a_raw, b_raw, normalize_q, norm_eps):
        q, k, alpha, beta = prep(k_raw, a_raw, b_raw, q_raw=q_raw, normalize_q=normalize_q,
                                 norm_eps=norm_eps)
        ctx.save_for_backward(q_raw, k_raw, a_raw, b_raw)
        ctx.normalize_q, ctx.norm_eps = normalize_q, norm_eps
        return q, k, alpha, beta

    @staticmethod
    def backward(ctx, dq, dk, dalpha, dbeta):
        q_raw, k_raw, a_raw, b_raw = ctx.saved_tensors
        z = lambda g, like: torch.zeros_like(like) if g is None else g.contiguous()
        dq_raw, dk_raw, da_raw, db_raw = prep_bwd(
            k_raw, a_raw, b_raw, z(dk, k_raw), z(dalpha, a_raw), z(dbeta, b_raw), q_raw=q_raw,
            d_q=z(dq, q_raw), normalize_q=ctx.normalize_q, norm_eps=ctx.norm_eps)
        return dq_raw, dk_raw, da_raw, db_raw, None, None


def prepare(q_raw, k_raw, a_raw, b_raw, normalize_q=True, norm_eps=1e-6):
    """(q, k, alpha, beta) = prep(...) with q_raw given, differentiable in the
    raw inputs (the gradients come from prep_bwd)."""
    return _Prepare.apply(q_raw, k_raw, a_raw, b_raw, bool(normalize_q), float(norm_eps))
