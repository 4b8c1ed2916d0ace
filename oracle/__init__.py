"""fp64 CPU oracle for the Complex KDA (CKDA) recurrence -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.

The arithmetic lives in ``ckda_oracle.c`` (plain C, fp64, token by token, in
the order of "Kimi Delta Attention: a bounded case study", worked case A/B:
decay, read, correct, then read out the updated state as on the "Complex KDA"
discussion slides, frame "CKDA keeps the original gate--delta--readout
structure").  This module compiles it with gcc and marshals numpy arrays.

Functions and what pins them (tests/test_oracle_pins.py):

* ``fwd`` -- pinned by the worked decay/correction trace (bounded case study,
  worked case A and B), the one-step rotation R_{pi/2} (discussion slides,
  "Two reflections make a rotation in one update"), the closed form of Eq. (2)
  and the one-layer clock of Lemma 24 (paper), the Prop. 2 block, the
  non-expansiveness bound, the spectrum rule of Thm. 8, orthogonality of
  signed Householder products (Thm. 1), brute-force products of explicit
  n x n transition matrices, the sign gauge, channel permutations and the
  exact-retrieval reduction.
* ``decode_step`` -- pinned against ``fwd`` token by token and by the same
  rotation/decay fixtures.
* ``bwd`` -- reverse-mode gradients of sum <o, do> + <hT, dhT>: pinned by
  central finite differences of ``fwd`` (itself pinned above) on small
  problems, including gates exactly 0 and -1 and beta = 2, and by the
  closed form of the gradients when beta = 0 and alpha = 1 (o_t = h0^T q_t).
* ``prep`` -- the gate parameterisation and key normalisation ("Complex KDA"
  discussion slides, backup frame "practical gates differ from exact
  theoretical endpoints"): pinned by the properties that frame states (sign
  rule with s = +1 at r = 0, log|alpha| in [-5, 0], beta in (0, 2), the
  endpoints +-e^-5 next to a = 0 and |alpha| -> 1, beta -> 0 or 2 for large
  logits) and by the identities the parameterisation implies (odd symmetry of
  alpha, beta(-b) = 2 - beta(b), monotonicity in |a|, unit norm and direction
  of the normalised keys).
* ``prep_bwd`` -- the backward of ``prep``: pinned by central differences of
  ``prep`` (itself pinned above) away from a = 0, by the reading at a = 0
  (the sign carries no gradient, |r| takes the subgradient 0), by the closed
  form dbeta/db = 1/2 at b = 0, by the scale invariance of k / |k| (k_raw .
  dk_raw = 0 when norm_eps = 0) and by the identity map of an unnormalised q.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ckda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libckda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ckda_oracle.c into a shared library next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            lib.ckda_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, ip,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int]
            lib.ckda_oracle_fwd.restype = ctypes.c_int
            lib.ckda_oracle_decode_step.argtypes = [dp, dp, dp, dp, dp, dp, dp,
                                                    ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_double, ctypes.c_int]
            lib.ckda_oracle_decode_step.restype = ctypes.c_int
            lib.ckda_oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                            dp, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int]
            lib.ckda_oracle_bwd.restype = ctypes.c_int
            lib.ckda_oracle_prep.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_long,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_double]
            lib.ckda_oracle_prep.restype = ctypes.c_int
            lib.ckda_oracle_prep_bwd.argtypes = [dp] * 12 + [ctypes.c_long, ctypes.c_int,
                                                             ctypes.c_int, ctypes.c_double]
            lib.ckda_oracle_prep_bwd.restype = ctypes.c_int
            lib.ckda_oracle_max_threads.argtypes = []
            lib.ckda_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen exactly on the CPU
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().ckda_oracle_max_threads())


def fwd(q, k, v, alpha, beta, h0=None, cu_seqlens=None, scale=1.0,
        store_o=True, store_hT=True, nthreads=0):
    """Token-by-token fp64 recurrence.

    q, k, alpha: [B, H, T, dk]; v: [B, H, T, dv]; beta: [B, H, T];
    h0: [N, H, dk, dv] or None (zero state); cu_seqlens: [N + 1] int or None.
    Returns (o [B,H,T,dv] or None, hT [N,H,dk,dv] or None) as fp64 numpy.
    """
    lib = _load()
    q, k, v, alpha, beta, h0 = (_f64(a) for a in (q, k, v, alpha, beta, h0))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    cu = None
    N = B
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = cu.shape[0] - 1
    o = np.zeros((B, H, T, dv), dtype=np.float64) if store_o else None
    hT = np.zeros((N, H, dk, dv), dtype=np.float64) if store_hT else None
    rc = lib.ckda_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                             _ptr(h0), _ptr(o), _ptr(hT),
                             None if cu is None else cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                             int(N if cu is not None else 0), B, H, T, dk, dv,
                             float(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle fwd: invalid arguments")
    return o, hT


def decode_step(q, k, v, alpha, beta, state, scale=1.0, nthreads=0):
    """One token on a resident state.  Returns (o [B,H,dv], new_state)."""
    lib = _load()
    q, k, v, alpha, beta = (_f64(a) for a in (q, k, v, alpha, beta))
    S = _f64(state).copy()
    B, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, dv), dtype=np.float64)
    rc = lib.ckda_oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                     _ptr(S), _ptr(o), B, H, dk, dv, float(scale),
                                     int(nthreads))
    if rc != 0:
        raise ValueError("oracle decode_step: invalid arguments")
    return o, S


def prep(k_raw, a_raw, b_raw, q_raw=None, normalize_q=True, norm_eps=1e-6):
    """Input preparation in fp64: (q, k, alpha, beta) from raw q, k and the gate
    logits a [.., dk] and b [..] (q is None when q_raw is None)."""
    lib = _load()
    k_raw, a_raw, b_raw, q_raw = (_f64(x) for x in (k_raw, a_raw, b_raw, q_raw))
    dk = k_raw.shape[-1]
    rows = k_raw.size // dk
    if a_raw.shape != k_raw.shape or b_raw.size != rows or (
            q_raw is not None and q_raw.shape != k_raw.shape):
        raise ValueError("oracle prep: shapes")
    k = np.zeros_like(k_raw)
    alpha = np.zeros_like(a_raw)
    beta = np.zeros(b_raw.shape, dtype=np.float64)
    q = None if q_raw is None else np.zeros_like(q_raw)
    rc = lib.ckda_oracle_prep(_ptr(q_raw), _ptr(k_raw), _ptr(a_raw), _ptr(b_raw), _ptr(q),
                              _ptr(k), _ptr(alpha), _ptr(beta), int(rows), int(dk),
                              int(bool(normalize_q)), float(norm_eps))
    if rc != 0:
        raise ValueError("oracle prep: invalid arguments")
    return q, k, alpha, beta


def prep_bwd(k_raw, a_raw, b_raw, dk, dalpha, dbeta, q_raw=None, dq=None, normalize_q=True,
             norm_eps=1e-6):
    """Backward of ``prep`` in fp64: the gradients with respect to (q_raw, k_raw,
    a_raw, b_raw) from those with respect to its outputs (q, k, alpha, beta).
    The gate's sign carries no gradient and |tanh(a/2)| takes the subgradient
    0 at a = 0.  Returns (dq_raw or None, dk_raw, da_raw, db_raw)."""
    lib = _load()
    k_raw, a_raw, b_raw, q_raw, dk, dalpha, dbeta, dq = (
        _f64(x) for x in (k_raw, a_raw, b_raw, q_raw, dk, dalpha, dbeta, dq))
    n = k_raw.shape[-1]
    rows = k_raw.size // n
    shp = k_raw.shape
    if (a_raw.shape != shp or dk.shape != shp or dalpha.shape != shp or b_raw.size != rows
            or dbeta.size != rows or (q_raw is None) != (dq is None)
            or (q_raw is not None and (q_raw.shape != shp or dq.shape != shp))):
        raise ValueError("oracle prep_bwd: shapes")
    dk_raw, da_raw = np.zeros_like(k_raw), np.zeros_like(a_raw)
    db_raw = np.zeros(b_raw.shape, dtype=np.float64)
    dq_raw = None if q_raw is None else np.zeros_like(q_raw)
    rc = lib.ckda_oracle_prep_bwd(_ptr(q_raw), _ptr(k_raw), _ptr(a_raw), _ptr(b_raw), _ptr(dq),
                                  _ptr(dk), _ptr(dalpha), _ptr(dbeta), _ptr(dq_raw),
                                  _ptr(dk_raw), _ptr(da_raw), _ptr(db_raw), int(rows), int(n),
                                  int(bool(normalize_q)), float(norm_eps))
    if rc != 0:
        raise ValueError("oracle prep_bwd: invalid arguments")
    return dq_raw, dk_raw, da_raw, db_raw


def bwd(q, k, v, alpha, beta, do, h0=None, dhT=None, cu_seqlens=None, scale=1.0,
        store_dh0=True, nthreads=0):
    """Gradients of L = sum_t <o_t, do_t> + <hT, dhT> (fp64 numpy).

    Returns (dq, dk, dv, dalpha, dbeta, dh0 or None) in the layouts of the
    inputs ([B, H, T, .] and [N, H, dk, dv])."""
    lib = _load()
    q, k, v, alpha, beta, do, h0, dhT = (_f64(a) for a in (q, k, v, alpha, beta, do, h0, dhT))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    cu = None
    N = B
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = cu.shape[0] - 1
    dq, dkk, dal = (np.zeros_like(q) for _ in range(3))
    dvv = np.zeros_like(v)
    dbe = np.zeros_like(beta)
    dh0 = np.zeros((N, H, dk, dv), dtype=np.float64) if store_dh0 else None
    rc = lib.ckda_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(h0),
                             _ptr(do), _ptr(dhT), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dal),
                             _ptr(dbe), _ptr(dh0),
                             None if cu is None else cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                             int(N if cu is not None else 0), B, H, T, dk, dv, float(scale),
                             int(nthreads))
    if rc != 0:
        raise ValueError("oracle bwd: invalid arguments or out of memory")
    return dq, dkk, dvv, dal, dbe, dh0
