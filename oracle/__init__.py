"""fp64 CPU oracle for exact causal softmax attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product (``long_context_causal_gb300``) never imports it and shares no code
with it: the two meet only through the seeded inputs of
``long_context_causal_gb300.inputs``.

The arithmetic lives in ``oracle.c`` (plain fp64 loops, OpenMP over rows); this
module compiles it with gcc and marshals numpy arrays.  What is computed, and
the passages it follows, is documented at the top of ``oracle.c``:
DISTFLASHATTN (paperlayer.ai summary of arXiv 2310.03294) §3.1, §3.2, §3.3 and
App. D, with the online-normalizer merge rule of "Online normalizer
calculation for softmax".  ``attn_fwd_varlen`` / ``attn_bwd_varlen`` apply
the same definition to a packed batch of sequences of different lengths, one
sequence at a time (no token attends across a sequence boundary).

Parity status: every function here is pinned by ``tests/test_oracle.py``
(finite differences, closed forms, invariants, a library special case and
worked fixtures under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_I64 = ctypes.c_int64
_DP = ctypes.POINTER(ctypes.c_double)
_LP = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, fp64, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dims = [_I64] * 8 + [ctypes.c_int, ctypes.c_double]
            lib.oracle_fwd.argtypes = [_DP, _DP, _DP] + dims + [_DP, _DP, ctypes.c_int]
            lib.oracle_fwd_rows.argtypes = [_DP, _DP, _DP] + dims + [_LP, _I64, _DP, _DP, ctypes.c_int]
            lib.oracle_bwd.argtypes = [_DP, _DP, _DP, _DP] + dims + [_DP, _DP, _DP, ctypes.c_int]
            lib.oracle_dq_rows.argtypes = [_DP, _DP, _DP, _DP] + dims + [_LP, _I64, _DP, ctypes.c_int]
            lib.oracle_dkv_rows.argtypes = [_DP, _DP, _DP, _DP] + dims + [_LP, _I64, _DP, _DP, ctypes.c_int]
            lib.oracle_merge.argtypes = [_DP, _DP, _DP, _DP, _I64, _I64, _I64, _I64, _DP, _DP]
            local = [_I64] * 8 + [ctypes.c_double, _I64, _I64]
            lib.oracle_fwd_local.argtypes = [_DP, _DP, _DP] + local + [_DP, _DP, ctypes.c_int]
            lib.oracle_bwd_local.argtypes = [_DP, _DP, _DP, _DP] + local + [_DP, _DP, _DP, ctypes.c_int]
            lib.oracle_delta.argtypes = [_DP, _DP, _DP, _DP] + dims + [_DP, ctypes.c_int]
            lib.oracle_chunk_bwd.argtypes = [_DP, _DP, _DP, _DP, _DP, _DP] + dims + [_DP, _DP, _DP, ctypes.c_int]
            for f in ("oracle_fwd", "oracle_fwd_rows", "oracle_bwd", "oracle_dq_rows",
                      "oracle_dkv_rows", "oracle_merge", "oracle_num_threads", "oracle_delta",
                      "oracle_chunk_bwd", "oracle_fwd_local", "oracle_bwd_local"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses by default on this host."""
    return int(_load().oracle_num_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_DP)


def _dims(q, k, H_kv=None):
    B, Lq, H, D = q.shape
    Bk, Lkv, Hkv, Dk = k.shape
    assert B == Bk and D == Dk
    return B, H, Hkv, Lq, Lkv, D


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def attn_fwd(q, k, v, *, causal=True, scale=None, q_offset=0, kv_offset=0, threads=0):
    """O [B,Lq,H,D], lse [B,H,Lq] (natural log) in fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, Lq, Lkv, D = _dims(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    O = np.empty((B, Lq, H, D))
    lse = np.empty((B, H, Lq))
    rc = _load().oracle_fwd(_p(q), _p(k), _p(v), B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset,
                            int(bool(causal)), scale, _p(O), _p(lse), int(threads))
    _check(rc, "fwd")
    return O, lse


def attn_fwd_rows(q, k, v, rows, *, causal=True, scale=None, q_offset=0, kv_offset=0, threads=0):
    """O and lse on selected (b, h, i) query rows: returns ([n, D], [n])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, Lq, Lkv, D = _dims(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    O = np.empty((n, D))
    lse = np.empty((n,))
    rc = _load().oracle_fwd_rows(_p(q), _p(k), _p(v), B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset,
                                 int(bool(causal)), scale, rows.ctypes.data_as(_LP), n,
                                 _p(O), _p(lse), int(threads))
    _check(rc, "fwd_rows")
    return O, lse


def attn_bwd(q, k, v, dO, *, causal=True, scale=None, q_offset=0, kv_offset=0, threads=0):
    """dQ, dK, dV in fp64 from the explicit gradient formulas."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, Hkv, Lq, Lkv, D = _dims(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    dQ = np.empty_like(q)
    dK = np.empty_like(k)
    dV = np.empty_like(v)
    rc = _load().oracle_bwd(_p(q), _p(k), _p(v), _p(dO), B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset,
                            int(bool(causal)), scale, _p(dQ), _p(dK), _p(dV), int(threads))
    _check(rc, "bwd")
    return dQ, dK, dV


def attn_dq_rows(q, k, v, dO, rows, *, causal=True, scale=None, q_offset=0, kv_offset=0, threads=0):
    """dQ on selected (b, h, i) query rows: [n, D]."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, Hkv, Lq, Lkv, D = _dims(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.empty((rows.shape[0], D))
    rc = _load().oracle_dq_rows(_p(q), _p(k), _p(v), _p(dO), B, H, Hkv, Lq, Lkv, D, q_offset,
                                kv_offset, int(bool(causal)), scale, rows.ctypes.data_as(_LP),
                                rows.shape[0], _p(out), int(threads))
    _check(rc, "dq_rows")
    return out


def attn_dkv_rows(q, k, v, dO, krows, *, causal=True, scale=None, q_offset=0, kv_offset=0, threads=0):
    """dK, dV on selected (b, g, j) key rows: ([n, D], [n, D])."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, Hkv, Lq, Lkv, D = _dims(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    krows = np.ascontiguousarray(np.asarray(krows, dtype=np.int64).reshape(-1, 3))
    n = krows.shape[0]
    dK = np.empty((n, D))
    dV = np.empty((n, D))
    rc = _load().oracle_dkv_rows(_p(q), _p(k), _p(v), _p(dO), B, H, Hkv, Lq, Lkv, D, q_offset,
                                 kv_offset, int(bool(causal)), scale, krows.ctypes.data_as(_LP), n,
                                 _p(dK), _p(dV), int(threads))
    _check(rc, "dkv_rows")
    return dK, dV


def attn_fwd_local(q, k, v, *, chunk, window, scale=None, q_offset=0, kv_offset=0, threads=0):
    """Causal forward where a query sees only its own chunk (chunk tokens long,
    positions counted from 0) and the window - 1 chunks before it."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, Lq, Lkv, D = _dims(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    O = np.empty_like(q)
    lse = np.empty((B, H, Lq))
    rc = _load().oracle_fwd_local(_p(q), _p(k), _p(v), B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, scale,
                                  int(chunk), int(window), _p(O), _p(lse), int(threads))
    _check(rc, "fwd_local")
    return O, lse


def attn_bwd_local(q, k, v, dO, *, chunk, window, scale=None, q_offset=0, kv_offset=0, threads=0):
    """dQ, dK, dV of attn_fwd_local."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, Hkv, Lq, Lkv, D = _dims(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    dQ, dK, dV = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    rc = _load().oracle_bwd_local(_p(q), _p(k), _p(v), _p(dO), B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset,
                                  scale, int(chunk), int(window), _p(dQ), _p(dK), _p(dV), int(threads))
    _check(rc, "bwd_local")
    return dQ, dK, dV


def delta(q, k, v, dO, *, causal=True, scale=None, q_offset=0, kv_offset=0, threads=0):
    """Delta [B,H,Lq] = sum_j P_ij dP_ij over each row's visible keys, fp64."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, Hkv, Lq, Lkv, D = _dims(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.empty((B, H, Lq))
    rc = _load().oracle_delta(_p(q), _p(k), _p(v), _p(dO), B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset,
                              int(bool(causal)), scale, _p(out), int(threads))
    _check(rc, "delta")
    return out


def chunk_bwd(q, k, v, dO, lse, dlt, *, causal=True, scale=None, q_offset=0, kv_offset=0, threads=0):
    """Backward of one (query chunk, key chunk) pair given the rows' global lse
    and Delta [B,H,Lq]: partial dQ [B,Lq,H,D] (this chunk's keys), partial dK, dV
    [B,Lkv,H_kv,D] (this chunk's queries), fp64."""
    q, k, v, dO, lse, dlt = _f64(q), _f64(k), _f64(v), _f64(dO), _f64(lse), _f64(dlt)
    B, H, Hkv, Lq, Lkv, D = _dims(q, k)
    assert lse.shape == (B, H, Lq) and dlt.shape == (B, H, Lq)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    dQ = np.empty_like(q)
    dK = np.empty_like(k)
    dV = np.empty_like(v)
    rc = _load().oracle_chunk_bwd(_p(q), _p(k), _p(v), _p(dO), _p(lse), _p(dlt), B, H, Hkv, Lq, Lkv, D,
                                  q_offset, kv_offset, int(bool(causal)), scale, _p(dQ), _p(dK), _p(dV),
                                  int(threads))
    _check(rc, "chunk_bwd")
    return dQ, dK, dV


def merge(O_a, lse_a, O_b, lse_b):
    """Rescale-and-merge of two partials: O [B,L,H,D], lse [B,H,L]."""
    O_a, lse_a, O_b, lse_b = _f64(O_a), _f64(lse_a), _f64(O_b), _f64(lse_b)
    B, L, H, D = O_a.shape
    O = np.empty_like(O_a)
    lse = np.empty_like(lse_a)
    rc = _load().oracle_merge(_p(O_a), _p(lse_a), _p(O_b), _p(lse_b), B, H, L, D, _p(O), _p(lse))
    _check(rc, "merge")
    return O, lse


def _cu(cu_seqlens, T):
    cu = np.asarray(cu_seqlens, dtype=np.int64).reshape(-1)
    if cu.size < 1 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, never decrease and end at the packed length")
    return cu


def attn_fwd_varlen(q, k, v, cu_seqlens, *, causal=True, scale=None, threads=0):
    """Variable-length batch packed along the token axis: q [T, H, D], k, v
    [T, H_kv, D]; sequence s holds tokens [cu[s], cu[s+1]) and attends only to
    its own tokens (causal inside the sequence when causal).  Returns O [T, H, D]
    and lse [H, T].  Attention of one sequence never reads another, so the
    result is the plain attention of every sequence on its own."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, D = q.shape
    cu = _cu(cu_seqlens, T)
    O = np.zeros_like(q)
    lse = np.zeros((H, T))
    for s in range(cu.size - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if a == b:
            continue
        Os, ls = attn_fwd(q[None, a:b], k[None, a:b], v[None, a:b], causal=causal, scale=scale, threads=threads)
        O[a:b] = Os[0]
        lse[:, a:b] = ls[0]
    return O, lse


def attn_bwd_varlen(q, k, v, dO, cu_seqlens, *, causal=True, scale=None, threads=0):
    """dQ [T, H, D], dK, dV [T, H_kv, D] of attn_fwd_varlen."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    T = q.shape[0]
    cu = _cu(cu_seqlens, T)
    dQ, dK, dV = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s in range(cu.size - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if a == b:
            continue
        g = attn_bwd(q[None, a:b], k[None, a:b], v[None, a:b], dO[None, a:b], causal=causal, scale=scale,
                     threads=threads)
        dQ[a:b], dK[a:b], dV[a:b] = g[0][0], g[1][0], g[2][0]
    return dQ, dK, dV
