"""Python binding of libdfa.so (include/dfa.h) -- argument marshalling only.

Each function has the name of the C entry point it calls.  Torch tensors are
used for device memory and streams: the binding reads their data pointers,
sizes and strides, allocates missing outputs/workspace with torch, passes the
current CUDA stream, and raises ``DfaError`` on any non-OK status.  All
arithmetic runs in the library's CUDA kernels; there is no CPU fallback, and
importing this module fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# DFA_LIB_PATH selects another build of the same library (e.g. a profiling build).
LIB_PATH = os.environ.get("DFA_LIB_PATH") or os.path.join(_PKG, "libdfa.so")
INCLUDE = os.path.join(os.path.dirname(_PKG), "include")
HEADER = os.path.join(INCLUDE, "dfa.h")

DFA_OK, DFA_ERR_INVALID_ARG, DFA_ERR_UNSUPPORTED, DFA_ERR_CUDA, DFA_ERR_TIMEOUT, DFA_ERR_WORKSPACE = range(6)
DFA_F32, DFA_BF16 = 0, 1
DFA_SCHED_BALANCED, DFA_SCHED_UNBALANCED, DFA_SCHED_SPLIT_KV = 0, 1, 2
KERNEL_KINDS = {"fwd": 0, "bwd": 1, "merge": 2, "delta": 3, "convert": 4, "copy": 5}
_SCHED = {"balanced": DFA_SCHED_BALANCED, "unbalanced": DFA_SCHED_UNBALANCED, "split_kv": DFA_SCHED_SPLIT_KV,
          DFA_SCHED_BALANCED: DFA_SCHED_BALANCED, DFA_SCHED_UNBALANCED: DFA_SCHED_UNBALANCED,
          DFA_SCHED_SPLIT_KV: DFA_SCHED_SPLIT_KV}


class DfaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dfa status {status}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    p64 = ctypes.POINTER(ctypes.c_int64)
    p32 = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "dfa_chunk_attn_fwd": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, p64, p64, i64, i64, i32, f32, vp, vp, vp]),
        "dfa_merge_partials": (i32, [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]),
        "dfa_attn_workspace_size": (sz, [i32, i32, i32, i32, i32, i32, i32]),
        "dfa_attn_fwd": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32, vp, vp, vp, sz, vp]),
        "dfa_attn_bwd": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                               vp, vp, vp, vp, sz, vp]),
        "dfa_chunk_attn_bwd": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i64, i64, i32, f32,
                                     vp, vp, vp, vp, sz, vp]),
        "dfa_chunk_bwd_workspace_size": (sz, [i32, i32, i32, i32, i32, i32]),
        "dfa_attn_fwd_local": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32, vp, vp, vp, sz, vp]),
        "dfa_attn_bwd_local": (i32, [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                     vp, vp, vp, vp, sz, vp]),
        "dfa_attn_fwd_noalloc": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32, vp, vp, vp]),
        "dfa_check_errors": (i32, [vp]),
        "dfa_shutdown": (None, []),
        "dfa_last_error": (ctypes.c_char_p, []),
        "dfa_launch_count": (i64, [i32]),
        "dfa_copy": (i32, [vp, vp, ctypes.c_size_t, vp]),
        "dfa_build_worklist": (i64, [i32, i32, i32, i32, p32, p32]),
        "dfa_chunk_schedule": (i32, [i32, i32, i32, p32]),
        "dfa_split_piece_tiles": (i32, [i32, i32, i32, i32, i32]),
        "dfa_build_varlen_worklist": (i64, [i32, p32, i32, i32, i32, i32, p32, p32]),
        "dfa_split_bwd_piece_tiles": (i32, [i32, i32, i32, i32, i32]),
        "dfa_build_bwd_split_worklist": (i64, [i32, i32, i32, i32, i32, p32, p32]),
        "dfa_attn_varlen_workspace_size": (sz, [p32, i32, i32, i32, i32, i32]),
        "dfa_attn_fwd_varlen": (i32, [vp, vp, vp, i32, p32, i32, i32, i32, i32, i32, f32, vp, vp, vp, sz, vp]),
        "dfa_attn_bwd_varlen": (i32, [vp, vp, vp, vp, vp, vp, i32, p32, i32, i32, i32, i32, i32, f32,
                                      vp, vp, vp, vp, sz, vp]),
        "dfa_build_split_worklist": (i64, [i32, i32, i32, i32, i32, i32, p32, p32]),
        "dfa_debug_mma": (i32, [i32, vp, vp, vp, vp]),
        "dfa_debug_cta_trace": (i32, [vp, i32]),
        "dfa_debug_wait_timeout": (i32, [vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


_lib = _load()


def header_functions() -> list[str]:
    """Names of every function the headers under include/ declare."""
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            with open(os.path.join(INCLUDE, h)) as f:
                text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
            names.update(re.findall(r"\b(dfa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def library() -> ctypes.CDLL:
    return _lib


def _check(status: int):
    if status != DFA_OK:
        raise DfaError(status, _lib.dfa_last_error().decode())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DFA_F32
    if t.dtype == torch.bfloat16:
        return DFA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dense(t: torch.Tensor, name: str):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (BSHD dense)")


def _like(t: torch.Tensor, name: str, shape, dtype, device):
    """A caller-supplied output must be dense and have exactly the shape, dtype
    and device the kernels write: a smaller or narrower tensor would be written
    past its end."""
    _dense(t, name)
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device:
        raise ValueError(f"{name} must be a {dtype} tensor of shape {tuple(shape)} on {device}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")
    return t


def _inputs(q, k, v, *rest):
    """q, k, v (and O, dO where given) share one device; k and v one shape."""
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    for t in (k, v) + tuple(x for x in rest if x is not None):
        if t.device != q.device:
            raise ValueError("all tensors must be on the same device")


# ---------------------------------------------------------------- entry points
def dfa_chunk_attn_fwd(q, k, v, q_offset: int = 0, kv_offset: int = 0, causal: bool = True,
                       scale: float | None = None, O_partial=None, lse=None, stream=None):
    """One chunk step: returns (O_partial fp32 [B,Lq,H,D], lse fp32 [B,H,Lq])."""
    B, Lq, H, D = q.shape
    _, Lkv, Hkv, _ = k.shape
    if k.stride() != v.stride() or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must share dtype and strides with each other (and dtype with q)")
    if q.stride(3) != 1 or k.stride(3) != 1:
        raise ValueError("the head dimension must be contiguous")
    scale = D ** -0.5 if scale is None else float(scale)
    _inputs(q, k, v)
    if O_partial is None:
        O_partial = torch.empty((B, Lq, H, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32, device=q.device)
    _like(O_partial, "O_partial", (B, Lq, H, D), torch.float32, q.device)
    _like(lse, "lse", (B, H, Lq), torch.float32, q.device)
    qs = (ctypes.c_int64 * 3)(q.stride(0), q.stride(1), q.stride(2))
    ks = (ctypes.c_int64 * 3)(k.stride(0), k.stride(1), k.stride(2))
    _check(_lib.dfa_chunk_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _dtype(q), B, H, Hkv, Lq, Lkv, D,
                                   qs, ks, int(q_offset), int(kv_offset), int(bool(causal)), scale,
                                   _ptr(O_partial), _ptr(lse), _stream(stream)))
    return O_partial, lse


def dfa_chunk_bwd_workspace_size(B, H, H_kv, Lq, Lkv, D) -> int:
    return int(_lib.dfa_chunk_bwd_workspace_size(B, H, H_kv, Lq, Lkv, D))


def dfa_chunk_attn_bwd(q, k, v, O, lse, dO, q_offset: int = 0, kv_offset: int = 0, causal: bool = True,
                       scale: float | None = None, dQ_acc=None, dK_acc=None, dV_acc=None,
                       workspace_buf=None, stream=None):
    """Backward step of one (query chunk, key chunk) pair from the rows' final
    (O, lse): adds the pair's share into fp32 accumulators (created zeroed when
    not given) and returns (dQ_acc [B,Lq,H,D], dK_acc, dV_acc [B,Lkv,H_kv,D])."""
    B, Lq, H, D = q.shape
    _, Lkv, Hkv, _ = k.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (O, "O"), (lse, "lse"), (dO, "dO")):
        _dense(t, n)
    scale = D ** -0.5 if scale is None else float(scale)
    f32 = dict(dtype=torch.float32, device=q.device)
    dQ_acc = torch.zeros((B, Lq, H, D), **f32) if dQ_acc is None else dQ_acc
    dK_acc = torch.zeros((B, Lkv, Hkv, D), **f32) if dK_acc is None else dK_acc
    dV_acc = torch.zeros((B, Lkv, Hkv, D), **f32) if dV_acc is None else dV_acc
    _inputs(q, k, v, O, dO, lse)
    _like(O, "O", q.shape, q.dtype, q.device)
    _like(dO, "dO", q.shape, q.dtype, q.device)
    _like(lse, "lse", (B, H, Lq), torch.float32, q.device)
    _like(dQ_acc, "dQ_acc", (B, Lq, H, D), torch.float32, q.device)
    _like(dK_acc, "dK_acc", (B, Lkv, Hkv, D), torch.float32, q.device)
    _like(dV_acc, "dV_acc", (B, Lkv, Hkv, D), torch.float32, q.device)
    if workspace_buf is None:
        workspace_buf = torch.empty(max(dfa_chunk_bwd_workspace_size(B, H, Hkv, Lq, Lkv, D), 16),
                                    dtype=torch.uint8, device=q.device)
    _check(_lib.dfa_chunk_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(O), _ptr(lse), _ptr(dO), _dtype(q),
                                   B, H, Hkv, Lq, Lkv, D, int(q_offset), int(kv_offset), int(bool(causal)),
                                   scale, _ptr(dQ_acc), _ptr(dK_acc), _ptr(dV_acc), _ptr(workspace_buf),
                                   workspace_buf.numel(), _stream(stream)))
    return dQ_acc, dK_acc, dV_acc


def dfa_merge_partials(O_a, lse_a, O_b, lse_b, O_out=None, lse_out=None, stream=None):
    """Rescale-and-merge; O_out/lse_out may alias the inputs."""
    B, L, H, D = O_a.shape
    for t, n in ((O_a, "O_a"), (O_b, "O_b"), (lse_a, "lse_a"), (lse_b, "lse_b")):
        _dense(t, n)
    for t, n in ((O_a, "O_a"), (O_b, "O_b")):
        _like(t, n, (B, L, H, D), torch.float32, O_a.device)
    for t, n in ((lse_a, "lse_a"), (lse_b, "lse_b")):
        _like(t, n, (B, H, L), torch.float32, O_a.device)
    O_out = torch.empty_like(O_a) if O_out is None else O_out
    lse_out = torch.empty_like(lse_a) if lse_out is None else lse_out
    _like(O_out, "O_out", (B, L, H, D), torch.float32, O_a.device)
    _like(lse_out, "lse_out", (B, H, L), torch.float32, O_a.device)
    _check(_lib.dfa_merge_partials(B, H, L, D, _ptr(O_a), _ptr(lse_a), _ptr(O_b), _ptr(lse_b),
                                   _ptr(O_out), _ptr(lse_out), _stream(stream)))
    return O_out, lse_out


def dfa_attn_workspace_size(B, H, H_kv, S, D, n_chunks, bwd) -> int:
    return int(_lib.dfa_attn_workspace_size(B, H, H_kv, S, D, n_chunks, int(bool(bwd))))


def workspace(B, H, H_kv, S, D, n_chunks, bwd, device="cuda"):
    n = dfa_attn_workspace_size(B, H, H_kv, S, D, n_chunks, bwd)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def dfa_attn_fwd(q, k, v, n_chunks: int = 1, causal: bool = True, scale: float | None = None,
                 sched="balanced", O=None, lse=None, workspace_buf=None, stream=None):
    """Whole-sequence forward: returns (O [B,S,H,D] in q's dtype, lse fp32 [B,H,S])."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dense(t, n)
    scale = D ** -0.5 if scale is None else float(scale)
    _inputs(q, k, v)
    O = torch.empty_like(q) if O is None else _like(O, "O", q.shape, q.dtype, q.device)
    lse = (torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None
           else _like(lse, "lse", (B, H, S), torch.float32, q.device))
    ws = workspace(B, H, Hkv, S, D, n_chunks, False, q.device) if workspace_buf is None else workspace_buf
    _check(_lib.dfa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _dtype(q), B, H, Hkv, S, D, int(n_chunks),
                             int(bool(causal)), scale, _SCHED[sched], _ptr(O), _ptr(lse), _ptr(ws),
                             ws.numel(), _stream(stream)))
    return O, lse


def _cu_host(cu_seqlens):
    """Host int32 copy of the sequence offsets (list, numpy array or tensor on any device)."""
    import numpy as np
    if isinstance(cu_seqlens, torch.Tensor):
        cu_seqlens = cu_seqlens.detach().cpu().numpy()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64).reshape(-1))
    if cu.size < 1 or np.any(cu < 0) or np.any(cu > 2**31 - 1):
        raise DfaError(DFA_ERR_INVALID_ARG, "cu_seqlens must hold n_seq + 1 int32 offsets")
    return cu.astype(np.int32)


def _check_packed(cu, T):
    if int(cu[-1]) != T:
        raise DfaError(DFA_ERR_INVALID_ARG, f"cu_seqlens ends at {int(cu[-1])}, the packed tensors hold {T} tokens")


def _p32(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def dfa_attn_varlen_workspace_size(cu_seqlens, H, H_kv, D, bwd) -> int:
    cu = _cu_host(cu_seqlens)
    return int(_lib.dfa_attn_varlen_workspace_size(_p32(cu), cu.size - 1, H, H_kv, D, int(bool(bwd))))


def varlen_workspace(cu_seqlens, H, H_kv, D, bwd, device="cuda"):
    n = dfa_attn_varlen_workspace_size(cu_seqlens, H, H_kv, D, bwd)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def dfa_attn_fwd_varlen(q, k, v, cu_seqlens, causal: bool = True, scale: float | None = None, O=None, lse=None,
                        workspace_buf=None, stream=None):
    """Packed batch forward: q [T,H,D], k, v [T,H_kv,D]; returns (O [T,H,D], lse fp32 [H,T])."""
    T, H, D = q.shape
    Hkv = k.shape[1]
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dense(t, n)
    cu = _cu_host(cu_seqlens)
    _check_packed(cu, T)
    scale = D ** -0.5 if scale is None else float(scale)
    _inputs(q, k, v)
    O = torch.empty_like(q) if O is None else _like(O, "O", q.shape, q.dtype, q.device)
    lse = (torch.empty((H, T), dtype=torch.float32, device=q.device) if lse is None
           else _like(lse, "lse", (H, T), torch.float32, q.device))
    ws = varlen_workspace(cu, H, Hkv, D, False, q.device) if workspace_buf is None else workspace_buf
    _check(_lib.dfa_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _dtype(q), _p32(cu), cu.size - 1, H, Hkv, D,
                                    int(bool(causal)), scale, _ptr(O), _ptr(lse), _ptr(ws), ws.numel(),
                                    _stream(stream)))
    return O, lse


def dfa_attn_bwd_varlen(q, k, v, O, lse, dO, cu_seqlens, causal: bool = True, scale: float | None = None,
                        dQ=None, dK=None, dV=None, workspace_buf=None, stream=None):
    """Packed batch backward from the saved (O, lse): returns (dQ, dK, dV)."""
    T, H, D = q.shape
    Hkv = k.shape[1]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (O, "O"), (lse, "lse"), (dO, "dO")):
        _dense(t, n)
    cu = _cu_host(cu_seqlens)
    _check_packed(cu, T)
    scale = D ** -0.5 if scale is None else float(scale)
    _inputs(q, k, v, O, dO, lse)
    _like(O, "O", q.shape, q.dtype, q.device)
    _like(dO, "dO", q.shape, q.dtype, q.device)
    _like(lse, "lse", (H, T), torch.float32, q.device)
    dQ = torch.empty_like(q) if dQ is None else _like(dQ, "dQ", q.shape, q.dtype, q.device)
    dK = torch.empty_like(k) if dK is None else _like(dK, "dK", k.shape, q.dtype, q.device)
    dV = torch.empty_like(v) if dV is None else _like(dV, "dV", v.shape, q.dtype, q.device)
    ws = varlen_workspace(cu, H, Hkv, D, True, q.device) if workspace_buf is None else workspace_buf
    _check(_lib.dfa_attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(O), _ptr(lse), _ptr(dO), _dtype(q),
                                    _p32(cu), cu.size - 1, H, Hkv, D, int(bool(causal)), scale,
                                    _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(), _stream(stream)))
    return dQ, dK, dV


def dfa_attn_fwd_noalloc(q, k, v, O, lse, n_chunks: int = 1, causal: bool = True,
                         scale: float | None = None, sched="balanced", stream=None):
    """dfa_attn_fwd without a workspace: writes the caller's O and lse, allocates nothing."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dense(t, n)
    _inputs(q, k, v)
    _like(O, "O", q.shape, q.dtype, q.device)
    _like(lse, "lse", (B, H, S), torch.float32, q.device)
    scale = D ** -0.5 if scale is None else float(scale)
    _check(_lib.dfa_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _dtype(q), B, H, Hkv, S, D, int(n_chunks),
                                     int(bool(causal)), scale, _SCHED[sched], _ptr(O), _ptr(lse),
                                     _stream(stream)))
    return O, lse


def dfa_attn_bwd(q, k, v, O, lse, dO, n_chunks: int = 1, causal: bool = True,
                 scale: float | None = None, sched="balanced", dQ=None, dK=None, dV=None,
                 workspace_buf=None, stream=None):
    """Backward from the saved (O, lse): returns (dQ, dK, dV) in q's dtype."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (O, "O"), (lse, "lse"), (dO, "dO")):
        _dense(t, n)
    scale = D ** -0.5 if scale is None else float(scale)
    _inputs(q, k, v, O, dO, lse)
    _like(O, "O", q.shape, q.dtype, q.device)
    _like(dO, "dO", q.shape, q.dtype, q.device)
    _like(lse, "lse", (B, H, S), torch.float32, q.device)
    dQ = torch.empty_like(q) if dQ is None else _like(dQ, "dQ", q.shape, q.dtype, q.device)
    dK = torch.empty_like(k) if dK is None else _like(dK, "dK", k.shape, q.dtype, q.device)
    dV = torch.empty_like(v) if dV is None else _like(dV, "dV", v.shape, q.dtype, q.device)
    ws = workspace(B, H, Hkv, S, D, n_chunks, True, q.device) if workspace_buf is None else workspace_buf
    _check(_lib.dfa_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(O), _ptr(lse), _ptr(dO), _dtype(q),
                             B, H, Hkv, S, D, int(n_chunks), int(bool(causal)), scale, _SCHED[sched],
                             _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(), _stream(stream)))
    return dQ, dK, dV


def dfa_attn_fwd_local(q, k, v, n_chunks: int, window: int, scale: float | None = None, sched="balanced",
                       O=None, lse=None, workspace_buf=None, stream=None):
    """Causal forward restricted to a local window of `window` chunks
    (ceil(S / n_chunks) tokens each, the last chunk possibly shorter): returns
    (O, lse) like dfa_attn_fwd."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dense(t, n)
    scale = D ** -0.5 if scale is None else float(scale)
    _inputs(q, k, v)
    O = torch.empty_like(q) if O is None else _like(O, "O", q.shape, q.dtype, q.device)
    lse = (torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None
           else _like(lse, "lse", (B, H, S), torch.float32, q.device))
    ws = workspace(B, H, Hkv, S, D, n_chunks, False, q.device) if workspace_buf is None else workspace_buf
    _check(_lib.dfa_attn_fwd_local(_ptr(q), _ptr(k), _ptr(v), _dtype(q), B, H, Hkv, S, D, int(n_chunks),
                                   int(window), scale, _SCHED[sched], _ptr(O), _ptr(lse), _ptr(ws), ws.numel(),
                                   _stream(stream)))
    return O, lse


def dfa_attn_bwd_local(q, k, v, O, lse, dO, n_chunks: int, window: int, scale: float | None = None,
                       sched="balanced", dQ=None, dK=None, dV=None, workspace_buf=None, stream=None):
    """Backward of dfa_attn_fwd_local from the saved (O, lse): returns (dQ, dK, dV)."""
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (O, "O"), (lse, "lse"), (dO, "dO")):
        _dense(t, n)
    scale = D ** -0.5 if scale is None else float(scale)
    _inputs(q, k, v, O, dO, lse)
    _like(O, "O", q.shape, q.dtype, q.device)
    _like(dO, "dO", q.shape, q.dtype, q.device)
    _like(lse, "lse", (B, H, S), torch.float32, q.device)
    dQ = torch.empty_like(q) if dQ is None else _like(dQ, "dQ", q.shape, q.dtype, q.device)
    dK = torch.empty_like(k) if dK is None else _like(dK, "dK", k.shape, q.dtype, q.device)
    dV = torch.empty_like(v) if dV is None else _like(dV, "dV", v.shape, q.dtype, q.device)
    ws = workspace(B, H, Hkv, S, D, n_chunks, True, q.device) if workspace_buf is None else workspace_buf
    _check(_lib.dfa_attn_bwd_local(_ptr(q), _ptr(k), _ptr(v), _ptr(O), _ptr(lse), _ptr(dO), _dtype(q),
                                   B, H, Hkv, S, D, int(n_chunks), int(window), scale, _SCHED[sched],
                                   _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(), _stream(stream)))
    return dQ, dK, dV


def dfa_debug_mma(form: int, A, B, C=None, stream=None):
    """One 128x128x128 tcgen05 product of the given operand form (include/dfa_debug.h)."""
    C = torch.empty((128, 128), dtype=torch.float32, device=A.device) if C is None else C
    _check(_lib.dfa_debug_mma(int(form), _ptr(A), _ptr(B), _ptr(C), _stream(stream)))
    return C


def dfa_debug_cta_trace(buf=None):
    """Turns the per-CTA timeline on (buf: int64 CUDA tensor of 16*n) or off (None)."""
    if buf is None:
        _check(_lib.dfa_debug_cta_trace(None, 0))
    else:
        _check(_lib.dfa_debug_cta_trace(_ptr(buf), buf.numel() // 16))
    return buf


def dfa_shutdown():
    """Releases the library's cached pinned work lists and staging buffers."""
    _lib.dfa_shutdown()


def dfa_debug_wait_timeout(out=None, stream=None):
    """Launches the bounded-wait timeout kernel (out: optional int32 CUDA tensor of 2)."""
    _check(_lib.dfa_debug_wait_timeout(_ptr(out), _stream(stream)))
    return out


def dfa_check_errors(stream=None):
    _check(_lib.dfa_check_errors(_stream(stream)))


def dfa_last_error() -> str:
    return _lib.dfa_last_error().decode()


def dfa_launch_count(kind: str | int) -> int:
    return int(_lib.dfa_launch_count(KERNEL_KINDS.get(kind, kind)))


def dfa_copy(dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
    """dst <- src, byte for byte, through the SMs (include/dfa.h: dfa_copy).
    Both dense, with the same byte count; each on the GPU or in pinned host
    memory.  Asynchronous on `stream` (default: the current stream)."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.numel() and not t.is_cuda and not t.is_pinned():   # an empty tensor has no memory to pin
            raise ValueError(f"{name} must be on the GPU or in pinned host memory")
    nb = dst.numel() * dst.element_size()
    if nb != src.numel() * src.element_size():
        raise ValueError(f"byte counts differ: dst {nb}, src {src.numel() * src.element_size()}")
    _check(_lib.dfa_copy(_ptr(dst), _ptr(src), nb, _stream(stream)))
    return dst


def dfa_build_worklist(n_rows: int, n_units: int, n_workers: int, sched="balanced"):
    """Host-only: returns (offsets list, items list, makespan in tiles)."""
    import numpy as np
    offsets = np.zeros(n_workers + 1, dtype=np.int32)
    items = np.zeros(max(n_rows * n_units, 1), dtype=np.int32)
    p32 = ctypes.POINTER(ctypes.c_int32)
    mk = _lib.dfa_build_worklist(n_rows, n_units, n_workers, _SCHED[sched],
                                 offsets.ctypes.data_as(p32), items.ctypes.data_as(p32))
    if mk < 0:
        raise DfaError(DFA_ERR_INVALID_ARG, "bad work-list arguments")
    return offsets, items[: n_rows * n_units], int(mk)


def dfa_split_piece_tiles(B: int, H: int, S: int, causal: bool, n_sms: int) -> int:
    """Host-only: the split-kv piece length (128-key tiles) for this problem, 0 if not split."""
    return int(_lib.dfa_split_piece_tiles(B, H, S, int(bool(causal)), n_sms))


def dfa_build_split_worklist(n_rows: int, n_units: int, kv_tiles: int, causal: bool, piece_tiles: int,
                             n_workers: int):
    """Host-only: split-kv pieces dealt to workers -> (offsets, items, makespan)."""
    import numpy as np
    n_split = max(1, -(-kv_tiles // piece_tiles)) if piece_tiles > 0 else 1
    offsets = np.zeros(n_workers + 1, dtype=np.int32)
    items = np.zeros(max(n_rows * n_units * n_split, 1), dtype=np.int32)
    p32 = ctypes.POINTER(ctypes.c_int32)
    mk = _lib.dfa_build_split_worklist(n_rows, n_units, kv_tiles, int(bool(causal)), piece_tiles, n_workers,
                                       offsets.ctypes.data_as(p32), items.ctypes.data_as(p32))
    if mk < 0:
        raise DfaError(DFA_ERR_INVALID_ARG, "bad split work-list arguments")
    return offsets, items[: offsets[-1]], int(mk)


def dfa_split_bwd_piece_tiles(B: int, H_kv: int, S: int, causal: bool, n_sms: int) -> int:
    """Host-only: the backward split-kv piece length (query tiles), 0 if not split."""
    return int(_lib.dfa_split_bwd_piece_tiles(B, H_kv, S, int(bool(causal)), n_sms))


def dfa_build_bwd_split_worklist(n_rows: int, kv_tiles: int, causal: bool, piece_tiles: int, n_workers: int):
    """Host-only: backward split-kv pieces dealt to workers -> (offsets, items, makespan)."""
    import numpy as np
    n_split = max(1, -(-kv_tiles // piece_tiles)) if piece_tiles > 0 else 1
    offsets = np.zeros(n_workers + 1, dtype=np.int32)
    items = np.zeros(max(n_rows * kv_tiles * n_split, 1), dtype=np.int32)
    mk = _lib.dfa_build_bwd_split_worklist(n_rows, kv_tiles, int(bool(causal)), piece_tiles, n_workers,
                                           _p32(offsets), _p32(items))
    if mk < 0:
        raise DfaError(DFA_ERR_INVALID_ARG, "bad backward split work-list arguments")
    return offsets, items[: offsets[-1]], int(mk)


def dfa_build_varlen_worklist(seq_units, heads: int, n_units_max: int, causal: bool, n_workers: int):
    """Host-only: packed-batch items dealt to workers -> (offsets, items, makespan)."""
    import numpy as np
    units = np.ascontiguousarray(np.asarray(seq_units, dtype=np.int32).reshape(-1))
    offsets = np.zeros(n_workers + 1, dtype=np.int32)
    items = np.zeros(max(units.size * heads * max(n_units_max, 1), 1), dtype=np.int32)
    mk = _lib.dfa_build_varlen_worklist(units.size, _p32(units), heads, n_units_max, int(bool(causal)), n_workers,
                                        _p32(offsets), _p32(items))
    if mk < 0:
        raise DfaError(DFA_ERR_INVALID_ARG, "bad packed-batch work-list arguments")
    return offsets, items[: offsets[-1]], int(mk)


def dfa_chunk_schedule(P: int, sched="balanced"):
    """Host-only: the per-step block schedule of P chunk workers -> int array [steps, P]."""
    import numpy as np
    cap = P + 1
    steps = np.zeros(cap * P, dtype=np.int32)
    n = _lib.dfa_chunk_schedule(P, _SCHED[sched], cap, steps.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    if n < 0:
        raise DfaError(DFA_ERR_INVALID_ARG, "bad chunk-schedule arguments")
    return steps[: n * P].reshape(n, P)
