"""ctypes binding of libdiffattn.so (the C ABI of include/diffattn.h).

Argument marshalling only: torch tensors supply device pointers, shapes and
the current CUDA stream; every step of the computation runs in the library's
kernels. There is no fallback of any kind: if the library is not built, or a
call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_BAD_SEQLENS, ERR_BAD_POSITIONS = range(7)
DTYPE_F32, DTYPE_BF16 = 0, 1

# Names the header declares with external linkage (checked by the ABI tests).
EXPORTED = ("diffattn_lambda_init", "diffattn_lambda", "diffattn_fwd", "diffattn_fwd_train",
            "diffattn_bwd_workspace_size", "diffattn_bwd", "diffattn_lambda_bwd", "diffattn_fwd_kvcache_workspace_size",
            "diffattn_fwd_kvcache", "diffattn_fwd_kvcache_noalloc", "diffattn_get_device_status",
            "diffattn_status_string", "diffattn_set_wait_timeout_ns", "diffattn_set_fault_injection",
            "diffattn_rope_tables", "diffattn_rope_qk", "diffattn_merge_partials", "diffattn_out_proj",
            "diffattn_fwd_kernel", "diffattn_fwd_rope_q", "diffattn_fwd_lambda", "diffattn_fwd_kvcache_lambda")


class DiffAttnDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("seqlen", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("max_seqlen", ctypes.c_int), ("total_tokens", ctypes.c_int), ("num_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("d", ctypes.c_int), ("dv", ctypes.c_int),
                ("dtype", ctypes.c_int), ("eps", ctypes.c_float)]


class DiffAttnKvDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("q_len", ctypes.c_int), ("cache_capacity", ctypes.c_int),
                ("num_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int), ("d", ctypes.c_int),
                ("dv", ctypes.c_int), ("dtype", ctypes.c_int), ("eps", ctypes.c_float), ("num_splits", ctypes.c_int),
                ("host_seqlens", ctypes.c_void_p)]


class DiffAttnRopeDesc(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_longlong), ("num_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("d", ctypes.c_int), ("dtype", ctypes.c_int), ("rot_dim", ctypes.c_int),
                ("interleaved", ctypes.c_int), ("n_pos", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("seqlen", ctypes.c_int)]


class DiffAttnRopeQ(ctypes.Structure):
    _fields_ = [("cos", ctypes.c_void_p), ("sin", ctypes.c_void_p), ("n_pos", ctypes.c_int), ("rot_dim", ctypes.c_int),
                ("interleaved", ctypes.c_int)]


class DiffAttnMergeDesc(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_longlong), ("num_heads", ctypes.c_int), ("dv", ctypes.c_int),
                ("n_parts", ctypes.c_int), ("out_dtype", ctypes.c_int), ("eps", ctypes.c_float)]


class DiffAttnOutProjDesc(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int), ("in_features", ctypes.c_int), ("out_features", ctypes.c_int)]


class DiffAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libdiffattn.so (built by `_build.build()` / `__graft_entry__.build()`)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libdiffattn.so is not built ({p}); run differential_attention_diffattn_gb300."
                               "_build.build() first")
        lib = ctypes.CDLL(p)
        vp, fp, ip = ctypes.c_void_p, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)
        lib.diffattn_lambda_init.restype = ctypes.c_float
        lib.diffattn_lambda_init.argtypes = [ctypes.c_int]
        lib.diffattn_lambda.restype = ctypes.c_int
        lib.diffattn_lambda.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_float, vp, vp]
        lib.diffattn_fwd_kernel.restype = ctypes.c_char_p
        lib.diffattn_fwd_kernel.argtypes = [ctypes.POINTER(DiffAttnDesc), ctypes.c_int]
        lib.diffattn_fwd_rope_q.restype = ctypes.c_int
        lib.diffattn_fwd_rope_q.argtypes = [ctypes.POINTER(DiffAttnDesc), vp, vp, vp, vp, ctypes.c_int, ctypes.c_float,
                                            vp, ctypes.c_int, vp, ctypes.POINTER(DiffAttnRopeQ), vp, vp]
        lib.diffattn_fwd_lambda.restype = ctypes.c_int
        lib.diffattn_fwd_lambda.argtypes = [ctypes.POINTER(DiffAttnDesc), vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_float, vp, vp, ctypes.c_int, vp, vp, vp]
        lib.diffattn_fwd.restype = ctypes.c_int
        lib.diffattn_fwd.argtypes = [ctypes.POINTER(DiffAttnDesc), vp, vp, vp, vp, ctypes.c_int, ctypes.c_float,
                                     vp, ctypes.c_int, vp, vp, vp]
        lib.diffattn_fwd_train.restype = ctypes.c_int
        lib.diffattn_fwd_train.argtypes = [ctypes.POINTER(DiffAttnDesc), vp, vp, vp, vp, ctypes.c_int, ctypes.c_float,
                                           vp, ctypes.c_int, vp, vp, vp, vp, vp, vp]
        lib.diffattn_bwd_workspace_size.restype = ctypes.c_ulonglong
        lib.diffattn_bwd_workspace_size.argtypes = [ctypes.POINTER(DiffAttnDesc)]
        lib.diffattn_bwd.restype = ctypes.c_int
        lib.diffattn_bwd.argtypes = [ctypes.POINTER(DiffAttnDesc), vp, vp, vp, vp, ctypes.c_int, ctypes.c_float, vp,
                                     ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_ulonglong, vp]
        lib.diffattn_lambda_bwd.restype = ctypes.c_int
        lib.diffattn_lambda_bwd.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp]
        lib.diffattn_fwd_kvcache_workspace_size.restype = ctypes.c_ulonglong
        lib.diffattn_fwd_kvcache_workspace_size.argtypes = [ctypes.POINTER(DiffAttnKvDesc)]
        lib.diffattn_fwd_kvcache.restype = ctypes.c_int
        lib.diffattn_fwd_kvcache.argtypes = [ctypes.POINTER(DiffAttnKvDesc), vp, vp, vp, vp, vp, ctypes.c_int,
                                             ctypes.c_float, vp, ctypes.c_int, vp, ctypes.c_ulonglong, vp, vp]
        lib.diffattn_fwd_kvcache_lambda.restype = ctypes.c_int
        lib.diffattn_fwd_kvcache_lambda.argtypes = [ctypes.POINTER(DiffAttnKvDesc), vp, vp, vp, vp, vp, vp, vp, vp,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_float, vp, vp, ctypes.c_int,
                                                    vp, ctypes.c_ulonglong, vp, vp]
        lib.diffattn_fwd_kvcache_noalloc.restype = ctypes.c_int
        lib.diffattn_fwd_kvcache_noalloc.argtypes = [ctypes.POINTER(DiffAttnKvDesc), vp, vp, vp, vp, vp, ctypes.c_int,
                                                     ctypes.c_float, vp, ctypes.c_int, vp, vp]
        lib.diffattn_get_device_status.restype = ctypes.c_int
        lib.diffattn_get_device_status.argtypes = [vp]
        lib.diffattn_status_string.restype = ctypes.c_char_p
        lib.diffattn_status_string.argtypes = [ctypes.c_int]
        lib.diffattn_set_wait_timeout_ns.restype = None
        lib.diffattn_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        lib.diffattn_set_fault_injection.restype = ctypes.c_int
        lib.diffattn_set_fault_injection.argtypes = [ctypes.c_int]
        lib.diffattn_rope_tables.restype = ctypes.c_int
        lib.diffattn_rope_tables.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int, vp, vp, vp]
        lib.diffattn_rope_qk.restype = ctypes.c_int
        lib.diffattn_rope_qk.argtypes = [ctypes.POINTER(DiffAttnRopeDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.diffattn_out_proj.restype = ctypes.c_int
        lib.diffattn_out_proj.argtypes = [ctypes.POINTER(DiffAttnOutProjDesc), vp, vp, vp, vp]
        lib.diffattn_merge_partials.restype = ctypes.c_int
        lib.diffattn_merge_partials.argtypes = [ctypes.POINTER(DiffAttnMergeDesc), vp, vp, vp, vp, ctypes.c_int,
                                                ctypes.c_float, vp, vp, vp]
        del fp, ip
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().diffattn_status_string(int(status)).decode()


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _check_cuda(t, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------- the ABI ---

def diffattn_lambda_init(depth: int) -> float:
    """lambda_init of layer `depth` (from 1), computed by the library (host)."""
    return float(load_library().diffattn_lambda_init(int(depth)))


def diffattn_lambda(lq1, lk1, lq2, lk2, lambda_init: float, out=None, stream=None):
    """lambda per parameter set on the GPU. Vectors fp32 [d] (one set) or
    [n, d] (n sets, e.g. per head); returns fp32 [n]."""
    import torch
    lib = load_library()
    vs = (lq1, lk1, lq2, lk2)
    for i, t in enumerate(vs):
        _check_cuda(t, f"lambda vector {i}")
        if t.dtype != torch.float32 or t.shape != lq1.shape:
            raise ValueError("lambda vectors must be fp32 of one shape")
    d = lq1.shape[-1]
    n = 1 if lq1.dim() == 1 else lq1.shape[0]
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=lq1.device)
    _check_cuda(out, "out")
    st = lib.diffattn_lambda(_ptr(lq1), _ptr(lk1), _ptr(lq2), _ptr(lk2), n, d, float(lambda_init), _ptr(out),
                             _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_lambda")
    return out


def diffattn_fwd_kernel(q, k, v, lam, subln_w, cu_seqlens=None, max_seqlen: Optional[int] = None,
                        eps: float = 1e-5) -> Optional[str]:
    """Name of the kernel diffattn_fwd / diffattn_fwd_train launch for these
    tensors (arguments as for diffattn_fwd; nothing is launched)."""
    desc, _ = _fwd_desc(q, k, v, lam, subln_w, cu_seqlens, max_seqlen, eps)
    name = load_library().diffattn_fwd_kernel(ctypes.byref(desc), 1 if cu_seqlens is not None else 0)
    return name.decode() if name else None


def _fwd_desc(q, k, v, lam, subln_w, cu_seqlens, max_seqlen, eps):
    """Checks shared by the forward entry points; returns (desc, H)."""
    import torch
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (lam, "lambda"), (subln_w, "subln_w")):
        _check_cuda(t, name)
    if q.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif q.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype")
    if lam.dtype != torch.float32 or subln_w.dtype != torch.float32:
        raise ValueError("lambda and subln_w must be fp32")
    desc = DiffAttnDesc()
    if q.dim() == 4:
        if cu_seqlens is not None:
            raise ValueError("cu_seqlens goes with token-major [tokens, H, 2d] inputs")
        B, T, H, two_d = q.shape
        desc.batch, desc.seqlen = B, T
    elif q.dim() == 3:
        tokens, H, two_d = q.shape
        if cu_seqlens is None:
            desc.batch, desc.seqlen = 1, tokens
        else:
            _check_cuda(cu_seqlens, "cu_seqlens")
            if cu_seqlens.dtype != torch.int32:
                raise ValueError("cu_seqlens must be int32")
            if max_seqlen is None:
                raise ValueError("max_seqlen is required with cu_seqlens")
            desc.num_seqs = cu_seqlens.numel() - 1
            desc.max_seqlen = int(max_seqlen)
            desc.total_tokens = tokens
    else:
        raise ValueError("q must be [B, T, H, 2d] or [tokens, H, 2d]")
    Hkv, dv = k.shape[-2], v.shape[-1]
    desc.num_heads, desc.num_kv_heads = H, Hkv
    desc.d, desc.dv = two_d // 2, dv
    desc.dtype = dt
    desc.eps = float(eps)
    if k.shape[:-2] != q.shape[:-2] or v.shape[:-2] != q.shape[:-2] or v.shape[-2] != Hkv:
        raise ValueError("q, k, v token dimensions or kv heads disagree")
    if lam.numel() not in (1, H):
        raise ValueError("lambda must hold 1 or H values")
    return desc, H


def diffattn_fwd_train(q, k, v, lam, lambda_init: float, subln_w, causal: bool = True, cu_seqlens=None,
                       max_seqlen: Optional[int] = None, eps: float = 1e-5, out=None, lse=None, o1=None, o2=None,
                       stream=None):
    """Forward that also returns what diffattn_bwd needs: (out, lse, o1, o2) with
    lse fp32 [..., H, 2] and o1, o2 fp32 [..., H, dv] (allocated when not given)."""
    import torch
    lib = load_library()
    desc, H = _fwd_desc(q, k, v, lam, subln_w, cu_seqlens, max_seqlen, eps)
    shp = q.shape[:-1]
    if out is None:
        out = torch.empty(shp + (v.shape[-1],), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(shp + (2,), dtype=torch.float32, device=q.device)
    if o1 is None:
        o1 = torch.empty(shp + (v.shape[-1],), dtype=torch.float32, device=q.device)
    if o2 is None:
        o2 = torch.empty_like(o1)
    for t, name in ((out, "out"), (lse, "lse"), (o1, "o1"), (o2, "o2")):
        _check_cuda(t, name)
    st = lib.diffattn_fwd_train(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(lam),
                                1 if (lam.numel() == H and H > 1) else 0, float(lambda_init), _ptr(subln_w),
                                1 if causal else 0, _ptr(cu_seqlens) if cu_seqlens is not None else None, _ptr(out),
                                _ptr(lse), _ptr(o1), _ptr(o2), _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_fwd_train")
    return out, lse, o1, o2


def diffattn_bwd_workspace_size(q, k, v, lam, subln_w, cu_seqlens=None, max_seqlen: Optional[int] = None,
                                eps: float = 1e-5) -> int:
    """Bytes of device scratch diffattn_bwd needs for these shapes."""
    desc, _ = _fwd_desc(q, k, v, lam, subln_w, cu_seqlens, max_seqlen, eps)
    return int(load_library().diffattn_bwd_workspace_size(ctypes.byref(desc)))


def diffattn_bwd(q, k, v, lam, lambda_init: float, subln_w, dout, lse, o1, o2, causal: bool = True,
                 cu_seqlens=None, max_seqlen: Optional[int] = None, eps: float = 1e-5, workspace=None,
                 grads=None, stream=None):
    """Gradients (dq, dk, dv, dlambda, dsubln_w) of diffattn_fwd_train's output;
    `grads` optionally gives those five tensors to write into."""
    import torch
    lib = load_library()
    desc, H = _fwd_desc(q, k, v, lam, subln_w, cu_seqlens, max_seqlen, eps)
    for t, name in ((dout, "dout"), (lse, "lse"), (o1, "o1"), (o2, "o2")):
        _check_cuda(t, name)
    need = int(lib.diffattn_bwd_workspace_size(ctypes.byref(desc)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if grads is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dlam = torch.empty(lam.numel() if (lam.numel() == H and H > 1) else 1, dtype=torch.float32,
                           device=q.device)
        dw = torch.empty_like(subln_w)
    else:
        dq, dk, dv, dlam, dw = grads
        for t, name in ((dq, "dq"), (dk, "dk"), (dv, "dv"), (dlam, "dlambda"), (dw, "dsubln_w")):
            _check_cuda(t, name)
    st = lib.diffattn_bwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(lam),
                          1 if (lam.numel() == H and H > 1) else 0, float(lambda_init), _ptr(subln_w),
                          1 if causal else 0, _ptr(cu_seqlens) if cu_seqlens is not None else None, _ptr(dout),
                          _ptr(lse), _ptr(o1), _ptr(o2), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dlam), _ptr(dw),
                          _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_bwd")
    return dq, dk, dv, dlam, dw


def diffattn_lambda_bwd(lq1, lk1, lq2, lk2, dlambda, stream=None):
    """Gradients of the four lambda vectors from the gradient of lambda."""
    import torch
    lib = load_library()
    d = lq1.shape[-1]
    n = 1 if lq1.dim() == 1 else lq1.shape[0]
    outs = [torch.empty_like(lq1) for _ in range(4)]
    st = lib.diffattn_lambda_bwd(_ptr(lq1), _ptr(lk1), _ptr(lq2), _ptr(lk2), _ptr(dlambda), n, d,
                                 *[_ptr(o) for o in outs], _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_lambda_bwd")
    return tuple(outs)


def _fwd_args(q, k, v, lam, subln_w, cu_seqlens, max_seqlen, eps, out):
    """Descriptor, head count and output tensor of a forward call (shared by
    diffattn_fwd and diffattn_fwd_rope_q)."""
    import torch
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (lam, "lambda"), (subln_w, "subln_w")):
        _check_cuda(t, name)
    if q.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif q.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype")
    if lam.dtype != torch.float32 or subln_w.dtype != torch.float32:
        raise ValueError("lambda and subln_w must be fp32")
    desc = DiffAttnDesc()
    if q.dim() == 4:
        if cu_seqlens is not None:
            raise ValueError("cu_seqlens goes with token-major [tokens, H, 2d] inputs")
        B, T, H, two_d = q.shape
        desc.batch, desc.seqlen = B, T
    elif q.dim() == 3:
        tokens, H, two_d = q.shape
        if cu_seqlens is None:
            desc.batch, desc.seqlen = 1, tokens
        else:
            _check_cuda(cu_seqlens, "cu_seqlens")
            if cu_seqlens.dtype != torch.int32:
                raise ValueError("cu_seqlens must be int32")
            if max_seqlen is None:
                raise ValueError("max_seqlen is required with cu_seqlens")
            desc.num_seqs = cu_seqlens.numel() - 1
            desc.max_seqlen = int(max_seqlen)
            desc.total_tokens = tokens
    else:
        raise ValueError("q must be [B, T, H, 2d] or [tokens, H, 2d]")
    Hkv, dv = k.shape[-2], v.shape[-1]
    desc.num_heads, desc.num_kv_heads = H, Hkv
    desc.d, desc.dv = two_d // 2, dv
    desc.dtype = dt
    desc.eps = float(eps)
    if k.shape[:-2] != q.shape[:-2] or v.shape[:-2] != q.shape[:-2] or v.shape[-2] != Hkv:
        raise ValueError("q, k, v token dimensions or kv heads disagree")
    if lam.numel() not in (1, H):
        raise ValueError("lambda must hold 1 or H values")
    if out is None:
        out = torch.empty(q.shape[:-1] + (dv,), dtype=q.dtype, device=q.device)
    _check_cuda(out, "out")
    return desc, H, out


def diffattn_fwd(q, k, v, lam, lambda_init: float, subln_w, causal: bool = True, cu_seqlens=None,
                 max_seqlen: Optional[int] = None, eps: float = 1e-5, out=None, stream=None):
    """Differential-attention forward on the GPU.

    q [B, T, H, 2d] with k [B, T, Hkv, 2d], v [B, T, Hkv, dv] (dense), or
    q [tokens, H, 2d] with k, v token-major and, for packed sequences,
    cu_seqlens int32 [num_seqs + 1] on the device plus max_seqlen (host int).
    lam: fp32 [1] (shared) or [H] (per head). Returns out [..., H, dv] in q's dtype.
    """
    lib = load_library()
    desc, H, out = _fwd_args(q, k, v, lam, subln_w, cu_seqlens, max_seqlen, eps, out)
    st = lib.diffattn_fwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(lam),
                          1 if (lam.numel() == H and H > 1) else 0, float(lambda_init), _ptr(subln_w),
                          1 if causal else 0, _ptr(cu_seqlens) if cu_seqlens is not None else None, _ptr(out),
                          _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_fwd")
    return out


def diffattn_fwd_lambda(q, k, v, lambda_q1, lambda_k1, lambda_q2, lambda_k2, lambda_init: float, subln_w,
                        causal: bool = True, cu_seqlens=None, max_seqlen: Optional[int] = None, eps: float = 1e-5,
                        lam_out=None, out=None, stream=None):
    """diffattn_lambda and diffattn_fwd in one call (the forward's loads and first
    tiles run while the lambda kernel finishes). lambda_q1 .. lambda_k2: fp32 [d]
    (shared lambda) or [H, d] (per head). Returns (out, lam)."""
    import torch
    lib = load_library()
    vecs = (lambda_q1, lambda_k1, lambda_q2, lambda_k2)
    for t, name in zip(vecs, ("lambda_q1", "lambda_k1", "lambda_q2", "lambda_k2")):
        _check_cuda(t, name)
        if t.dtype != torch.float32 or not t.is_contiguous() or t.shape != lambda_q1.shape:
            raise ValueError(f"{name} must be contiguous fp32 of the shape of lambda_q1")
    H = q.shape[-2]
    per_head = lambda_q1.dim() == 2 and lambda_q1.shape[0] == H and H > 1
    n_sets = H if per_head else 1
    if lam_out is None:
        lam_out = torch.empty(n_sets, dtype=torch.float32, device=q.device)
    _check_cuda(lam_out, "lam_out")
    desc, H, out = _fwd_args(q, k, v, lam_out, subln_w, cu_seqlens, max_seqlen, eps, out)
    st = lib.diffattn_fwd_lambda(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), *(_ptr(t) for t in vecs),
                                 1 if per_head else 0, int(lambda_q1.shape[-1]), float(lambda_init), _ptr(lam_out),
                                 _ptr(subln_w), 1 if causal else 0,
                                 _ptr(cu_seqlens) if cu_seqlens is not None else None, _ptr(out),
                                 _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_fwd_lambda")
    return out, lam_out


def diffattn_fwd_rope_q(q, k, v, lam, lambda_init: float, subln_w, cos, sin, rot_dim: int, interleaved: bool,
                        causal: bool = True, cu_seqlens=None, max_seqlen: Optional[int] = None, eps: float = 1e-5,
                        out=None, stream=None):
    """diffattn_fwd on q BEFORE its rotary embedding (the kernels rotate each
    query tile in shared memory; position = index inside the sequence); k must
    already be rotated (diffattn_rope_k). cos, sin: the tables of
    diffattn_rope_tables."""
    import torch
    lib = load_library()
    desc, H, out = _fwd_args(q, k, v, lam, subln_w, cu_seqlens, max_seqlen, eps, out)
    for t, name in ((cos, "cos"), (sin, "sin")):
        _check_cuda(t, name)
        if t.dtype != torch.float32:
            raise ValueError(f"{name} must be fp32")
    rope = DiffAttnRopeQ()
    rope.cos, rope.sin = _ptr(cos), _ptr(sin)
    rope.n_pos, rope.rot_dim, rope.interleaved = cos.shape[0], int(rot_dim), 1 if interleaved else 0
    st = lib.diffattn_fwd_rope_q(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(lam),
                                 1 if (lam.numel() == H and H > 1) else 0, float(lambda_init), _ptr(subln_w),
                                 1 if causal else 0, _ptr(cu_seqlens) if cu_seqlens is not None else None,
                                 ctypes.byref(rope), _ptr(out), _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_fwd_rope_q")
    return out


def kv_desc(q, k_cache, v_cache, eps: float = 1e-5, num_splits: int = 0, host_seqlens=None) -> DiffAttnKvDesc:
    """Descriptor of a cache forward from tensor shapes (q [B, q_len, H, 2d],
    k_cache [B, capacity, Hkv, 2d], v_cache [B, capacity, Hkv, dv]).
    host_seqlens: optional host copy of the cache lengths (a sequence of ints or
    a CPU tensor, [B]), which lets the library plan the key splits from them."""
    import torch
    if q.dim() != 4 or k_cache.dim() != 4 or v_cache.dim() != 4:
        raise ValueError("q, k_cache, v_cache must be 4-D")
    d = DiffAttnKvDesc()
    d.batch, d.q_len, d.num_heads = q.shape[0], q.shape[1], q.shape[2]
    d.cache_capacity, d.num_kv_heads = k_cache.shape[1], k_cache.shape[2]
    d.d, d.dv = q.shape[3] // 2, v_cache.shape[3]
    d.dtype = DTYPE_BF16 if q.dtype == torch.bfloat16 else DTYPE_F32
    d.eps, d.num_splits = float(eps), int(num_splits)
    d.host_seqlens = None
    if host_seqlens is not None:
        vals = [int(x) for x in (host_seqlens.tolist() if hasattr(host_seqlens, "tolist") else host_seqlens)]
        if len(vals) != d.batch:
            raise ValueError("host_seqlens must hold one length per sequence")
        arr = (ctypes.c_int * max(1, len(vals)))(*vals)
        d._host_arr = arr  # kept alive with the descriptor
        d.host_seqlens = ctypes.cast(arr, ctypes.c_void_p)
    return d


def diffattn_fwd_kvcache_workspace_size(desc: DiffAttnKvDesc) -> int:
    return int(load_library().diffattn_fwd_kvcache_workspace_size(ctypes.byref(desc)))


def diffattn_fwd_kvcache(q, k_cache, v_cache, lam, lambda_init: float, subln_w, cache_seqlens=None,
                         causal: bool = True, eps: float = 1e-5, num_splits: int = 0, workspace=None, out=None,
                         stream=None, host_seqlens=None):
    """New queries q [B, q_len, H, 2d] against a cache (k_cache [B, capacity,
    Hkv, 2d], v_cache [B, capacity, Hkv, dv], cache_seqlens int32 [B] on the
    device or None). The workspace (scratch for the key splits) is a caller
    buffer; when None the binding allocates one with torch for this call.
    host_seqlens: optional host copy of cache_seqlens for the split plan (a
    caller workspace must then be sized with the same lengths)."""
    import torch
    lib = load_library()
    for t, name in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (lam, "lambda"), (subln_w, "subln_w")):
        _check_cuda(t, name)
    if cache_seqlens is not None:
        _check_cuda(cache_seqlens, "cache_seqlens")
        if cache_seqlens.dtype != torch.int32 or cache_seqlens.numel() != q.shape[0]:
            raise ValueError("cache_seqlens must be int32 [batch]")
    desc = kv_desc(q, k_cache, v_cache, eps, num_splits, host_seqlens)
    need = int(lib.diffattn_fwd_kvcache_workspace_size(ctypes.byref(desc)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda(workspace, "workspace")
    if out is None:
        out = torch.empty(q.shape[:-1] + (v_cache.shape[-1],), dtype=q.dtype, device=q.device)
    _check_cuda(out, "out")
    H = q.shape[2]
    st = lib.diffattn_fwd_kvcache(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(cache_seqlens) if cache_seqlens is not None else None, _ptr(lam),
                                  1 if (lam.numel() == H and H > 1) else 0, float(lambda_init), _ptr(subln_w),
                                  1 if causal else 0, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _ptr(out), _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_fwd_kvcache")
    return out


def diffattn_fwd_kvcache_lambda(q, k_cache, v_cache, lambda_q1, lambda_k1, lambda_q2, lambda_k2, lambda_init: float,
                                subln_w, cache_seqlens=None, causal: bool = True, eps: float = 1e-5,
                                num_splits: int = 0, workspace=None, lam_out=None, out=None, stream=None,
                                host_seqlens=None):
    """diffattn_lambda and diffattn_fwd_kvcache in one call (the key-split kernel
    runs while the lambda kernel finishes; the combine kernel reads lambda).
    lambda_q1 .. lambda_k2: fp32 [d] (shared lambda) or [H, d] (per head).
    Returns (out, lam)."""
    import torch
    lib = load_library()
    vecs = (lambda_q1, lambda_k1, lambda_q2, lambda_k2)
    for t, name in zip(vecs, ("lambda_q1", "lambda_k1", "lambda_q2", "lambda_k2")):
        _check_cuda(t, name)
        if t.dtype != torch.float32 or not t.is_contiguous() or t.shape != lambda_q1.shape:
            raise ValueError(f"{name} must be contiguous fp32 of the shape of lambda_q1")
    for t, name in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (subln_w, "subln_w")):
        _check_cuda(t, name)
    if cache_seqlens is not None:
        _check_cuda(cache_seqlens, "cache_seqlens")
        if cache_seqlens.dtype != torch.int32 or cache_seqlens.numel() != q.shape[0]:
            raise ValueError("cache_seqlens must be int32 [batch]")
    H = q.shape[2]
    per_head = lambda_q1.dim() == 2 and lambda_q1.shape[0] == H and H > 1
    if lam_out is None:
        lam_out = torch.empty(H if per_head else 1, dtype=torch.float32, device=q.device)
    _check_cuda(lam_out, "lam_out")
    desc = kv_desc(q, k_cache, v_cache, eps, num_splits, host_seqlens)
    need = int(lib.diffattn_fwd_kvcache_workspace_size(ctypes.byref(desc)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_cuda(workspace, "workspace")
    if out is None:
        out = torch.empty(q.shape[:-1] + (v_cache.shape[-1],), dtype=q.dtype, device=q.device)
    _check_cuda(out, "out")
    st = lib.diffattn_fwd_kvcache_lambda(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(cache_seqlens) if cache_seqlens is not None else None,
                                         *(_ptr(t) for t in vecs), 1 if per_head else 0, int(lambda_q1.shape[-1]),
                                         float(lambda_init), _ptr(lam_out), _ptr(subln_w), 1 if causal else 0,
                                         _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
                                         _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_fwd_kvcache_lambda")
    return out, lam_out


def diffattn_fwd_kvcache_noalloc(q, k_cache, v_cache, lam, lambda_init: float, subln_w, cache_seqlens=None,
                                 causal: bool = True, eps: float = 1e-5, num_splits: int = 0, out=None,
                                 stream=None, host_seqlens=None):
    """diffattn_fwd_kvcache whose key-split scratch is the library's static device
    array instead of a workspace. The C entry point allocates nothing; only the
    output tensor is created here when `out` is None."""
    import torch
    lib = load_library()
    for t, name in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (lam, "lambda"), (subln_w, "subln_w")):
        _check_cuda(t, name)
    if cache_seqlens is not None:
        _check_cuda(cache_seqlens, "cache_seqlens")
        if cache_seqlens.dtype != torch.int32 or cache_seqlens.numel() != q.shape[0]:
            raise ValueError("cache_seqlens must be int32 [batch]")
    desc = kv_desc(q, k_cache, v_cache, eps, num_splits, host_seqlens)
    if out is None:
        out = torch.empty(q.shape[:-1] + (v_cache.shape[-1],), dtype=q.dtype, device=q.device)
    _check_cuda(out, "out")
    H = q.shape[2]
    st = lib.diffattn_fwd_kvcache_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(cache_seqlens) if cache_seqlens is not None else None, _ptr(lam),
                                          1 if (lam.numel() == H and H > 1) else 0, float(lambda_init),
                                          _ptr(subln_w), 1 if causal else 0, _ptr(out), _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_fwd_kvcache_noalloc")
    return out


def diffattn_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load_library().diffattn_get_device_status(_stream_handle(stream)))


def diffattn_status_string(status: int) -> str:
    return status_string(status)


def diffattn_set_wait_timeout_ns(ns: int) -> None:
    load_library().diffattn_set_wait_timeout_ns(int(ns))


def diffattn_set_fault_injection(mode: int) -> None:
    """Test hook of the failure-detection tests; the library honours it only in
    a process whose environment holds DIFFATTN_TEST_HOOKS=1."""
    st = load_library().diffattn_set_fault_injection(int(mode))
    if st != 0 and int(mode) != 0:
        raise DiffAttnError(st, "diffattn_set_fault_injection")


# ------------------------------------------------------------- rotary ---

def diffattn_rope_tables(theta: float, n_pos: int, rot_dim: int, device=None, stream=None):
    """(cos, sin) fp32 [n_pos, rot_dim/2] on the device: p * theta^(-2i/rot_dim),
    computed in fp64 by the kernel."""
    import torch
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    cos = torch.empty(n_pos, rot_dim // 2, dtype=torch.float32, device=dev)
    sin = torch.empty_like(cos)
    st = load_library().diffattn_rope_tables(float(theta), int(n_pos), int(rot_dim), _ptr(cos), _ptr(sin),
                                             _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_rope_tables")
    return cos, sin


def diffattn_rope_qk(q, k, cos, sin, rot_dim: int, interleaved: bool, positions=None, cu_seqlens=None,
                     q_out=None, k_out=None, stream=None):
    """Rotate q [tokens, H, 2d] (or [B, T, H, 2d]) and k (same layout with Hkv
    heads, or None); q may be None to rotate k only. Positions: `positions`
    int32 [tokens] if given, else `cu_seqlens` (packed sequences), else the
    dense layout. Pass q_out=q / k_out=k to rotate in place. Returns (q_out, k_out)."""
    import torch
    ref = q if q is not None else k
    if ref is None:
        raise ValueError("q or k is required")
    _check_cuda(ref, "q" if q is not None else "k")
    if ref.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif ref.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise ValueError(f"unsupported dtype {ref.dtype}")
    desc = DiffAttnRopeDesc()
    two_d = ref.shape[-1]
    desc.tokens = ref.numel() // (ref.shape[-2] * two_d)
    desc.num_heads, desc.d, desc.dtype = (q.shape[-2] if q is not None else 0), two_d // 2, dt
    desc.rot_dim, desc.interleaved = int(rot_dim), 1 if interleaved else 0
    desc.n_pos = cos.shape[0]
    if k is not None:
        _check_cuda(k, "k")
        if k.dtype != ref.dtype or k.shape[:-2] != ref.shape[:-2] or k.shape[-1] != two_d:
            raise ValueError("k must match q's dtype, token dims and head width")
        desc.num_kv_heads = k.shape[-2]
    for t, name in ((cos, "cos"), (sin, "sin")):
        _check_cuda(t, name)
        if t.dtype != torch.float32:
            raise ValueError(f"{name} must be fp32")
    if positions is not None:
        _check_cuda(positions, "positions")
        if positions.dtype != torch.int32 or positions.numel() != desc.tokens:
            raise ValueError("positions must be int32 [tokens]")
    elif cu_seqlens is not None:
        _check_cuda(cu_seqlens, "cu_seqlens")
        if cu_seqlens.dtype != torch.int32:
            raise ValueError("cu_seqlens must be int32")
        desc.num_seqs = cu_seqlens.numel() - 1
    else:
        desc.seqlen = ref.shape[1] if ref.dim() == 4 else ref.shape[0]
    if q is not None and q_out is None:
        q_out = torch.empty_like(q)
    if k is not None and k_out is None:
        k_out = torch.empty_like(k)
    st = load_library().diffattn_rope_qk(ctypes.byref(desc), _ptr(positions) if positions is not None else None,
                                         _ptr(cu_seqlens) if cu_seqlens is not None else None, _ptr(cos),
                                         _ptr(sin), _ptr(q) if q is not None else None,
                                         _ptr(q_out) if q is not None else None, _ptr(k) if k is not None else None,
                                         _ptr(k_out) if k is not None else None, _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_rope_qk")
    return q_out, k_out


def diffattn_rope_k(k, cos, sin, rot_dim: int, interleaved: bool, positions=None, cu_seqlens=None, k_out=None,
                    stream=None):
    """The rotary embedding of k alone (diffattn_rope_qk with num_heads = 0), the
    companion of diffattn_fwd_rope_q. Returns k_out."""
    return diffattn_rope_qk(None, k, cos, sin, rot_dim, interleaved, positions=positions, cu_seqlens=cu_seqlens,
                            k_out=k_out, stream=stream)[1]


# -------------------------------------------------------------- merge ---

def diffattn_merge_partials(lse, o1, o2, lam, lambda_init: float, subln_w, eps: float = 1e-5, out=None,
                            out_dtype=None, stream=None):
    """Merge stacked partials lse [n, ..., H, 2], o1 / o2 [n, ..., H, dv] (fp32,
    as diffattn_fwd_train saves them per key block) into the forward output
    [..., H, dv] (bf16 unless `out_dtype` or `out` says otherwise)."""
    import torch
    for t, name in ((lse, "lse"), (o1, "o1"), (o2, "o2"), (lam, "lambda"), (subln_w, "subln_w")):
        _check_cuda(t, name)
        if t.dtype != torch.float32:
            raise ValueError(f"{name} must be fp32")
    n, H, dv = o1.shape[0], o1.shape[-2], o1.shape[-1]
    if o2.shape != o1.shape or lse.shape[:-1] != o1.shape[:-1] or lse.shape[-1] != 2:
        raise ValueError("partials disagree in shape")
    if out is None:
        out = torch.empty(o1.shape[1:], dtype=out_dtype or torch.bfloat16, device=o1.device)
    _check_cuda(out, "out")
    desc = DiffAttnMergeDesc()
    desc.tokens = o1[0].numel() // (H * dv)
    desc.num_heads, desc.dv, desc.n_parts = H, dv, n
    desc.out_dtype = DTYPE_BF16 if out.dtype == torch.bfloat16 else DTYPE_F32
    desc.eps = float(eps)
    st = load_library().diffattn_merge_partials(ctypes.byref(desc), _ptr(lse), _ptr(o1), _ptr(o2), _ptr(lam),
                                                1 if (lam.numel() == H and H > 1) else 0, float(lambda_init),
                                                _ptr(subln_w), _ptr(out), _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_merge_partials")
    return out


# ----------------------------------------------------------- out_proj ---

def diffattn_out_proj(x, w, out=None, stream=None):
    """y = x W^T: w bf16 [N, K]; x bf16 contiguous with K values per row (e.g.
    the attention output [tokens, H, dv] or [B, T, H, dv] with K = H * dv).
    Returns y bf16 [rows, N], rows = x.numel() / K."""
    import torch
    for t, name in ((x, "x"), (w, "w")):
        _check_cuda(t, name)
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bf16")
    if w.dim() != 2:
        raise ValueError("w must be [N, K]")
    N, K = w.shape
    if x.numel() % K != 0:
        raise ValueError(f"x does not hold rows of {K} values")
    M = x.numel() // K
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _check_cuda(out, "out")
    desc = DiffAttnOutProjDesc()
    desc.tokens, desc.in_features, desc.out_features = M, K, N
    st = load_library().diffattn_out_proj(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(out), _stream_handle(stream))
    if st != OK:
        raise DiffAttnError(st, "diffattn_out_proj")
    return out
