"""Python side of the oracle for the differential-attention forward.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference arm, never by the product path. It shares
no code with the CUDA library.

Two independent fp64 statements of the same definition:

* `forward` / `forward_rows` call the C oracle (diffattn_oracle.c, built with
  gcc + OpenMP), which forms the two softmax-weighted value sums and subtracts
  them (the output-difference form of "LlamaDiffSdpaAttention.py", forward:
  attn1 - lambda_full * attn2);
* `forward_map_form` is a NumPy brute force that materialises both masked
  score maps, subtracts the probability maps and multiplies by V (the
  map-difference form of "DiffTransformer.py",
  MultiHeadDifferentialAttention.forward: attention1 - lambda_val * attention2,
  then matmul with V). It is for small cases only.

Both end with the per-head RMSNorm over dv, times the weight and (1 - lambda_init)
("DiffTransformer.py", forward, "Normalize each head independently using
RMSNorm" and "Scale the normalized output").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "diffattn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libdiffattn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP, no fast-math) if stale."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_lambda_init.restype = ctypes.c_double
    lib.oracle_lambda_init.argtypes = [ctypes.c_int]
    lib.oracle_lambda.restype = None
    lib.oracle_lambda.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_double, dp]
    lib.oracle_diffattn_rows.restype = ctypes.c_int
    lib.oracle_diffattn_rows.argtypes = [
        ctypes.c_int, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        dp, dp, dp, dp, ctypes.c_double, dp, ctypes.c_double, ctypes.c_int,
        ctypes.c_int, ip, ip, dp]
    return lib


def _load(path: Optional[str] = None):
    """The oracle library; `path` loads another build of the same source
    (the pin tests use this to check that planted mistakes are caught)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _f64(a) -> np.ndarray:
    """fp64 copy of a torch tensor or array (bf16 / fp32 values are exact in fp64)."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def num_threads() -> int:
    """Host threads the oracle's parallel loops run on."""
    return int(_load().oracle_num_threads())


def lambda_init(depth: int, lib=None) -> float:
    """0.8 - 0.6 exp(-0.3 (depth - 1)) ("DiffTransformer.py", DiffTransformer.__init__)."""
    return float((lib or _load()).oracle_lambda_init(int(depth)))


def lambda_values(lq1, lk1, lq2, lk2, lam_init: float, lib=None) -> np.ndarray:
    """exp(lq1.lk1) - exp(lq2.lk2) + lambda_init per parameter set
    ("DiffTransformer.py", forward, "Compute lambda using reparameterization").
    Vectors of shape [d] give one value; [n, d] give n values."""
    a = [_f64(x) for x in (lq1, lk1, lq2, lk2)]
    d = a[0].shape[-1]
    n = 1 if a[0].ndim == 1 else a[0].shape[0]
    a = [np.ascontiguousarray(x.reshape(n, d)) for x in a]
    out = np.zeros(n, dtype=np.float64)
    (lib or _load()).oracle_lambda(_dp(a[0]), _dp(a[1]), _dp(a[2]), _dp(a[3]), n, d, float(lam_init), _dp(out))
    return out


def _per_head_lambda(lam: np.ndarray, H: int) -> np.ndarray:
    lam = np.asarray(lam, dtype=np.float64).reshape(-1)
    if lam.size == 1:
        return np.full(H, lam[0], dtype=np.float64)
    if lam.size != H:
        raise ValueError(f"lambda has {lam.size} values for {H} heads")
    return np.ascontiguousarray(lam)


def forward_rows(cu_seqlens, q, k, v, lam, lam_init: float, w, eps: float, causal: bool,
                 rows: Optional[Sequence] = None, lib=None) -> np.ndarray:
    """C oracle. q [tokens, H, 2d], k [tokens, Hkv, 2d], v [tokens, Hkv, dv];
    `lam` holds one lambda (shared) or H values. With rows=None returns
    [tokens, H, dv]; with rows = (token_idx, head_idx) arrays returns [n, dv]."""
    cu = _i32(cu_seqlens)
    qa, ka, va, wa = _f64(q), _f64(k), _f64(v), _f64(w)
    tokens, H, two_d = qa.shape
    Hkv, dv = ka.shape[1], va.shape[2]
    d = two_d // 2
    lam_h = _per_head_lambda(lam, H)
    lib = lib or _load()
    if rows is None:
        out = np.zeros((tokens, H, dv), dtype=np.float64)
        n_rows, rt, rh = -1, np.zeros(1, np.int32), np.zeros(1, np.int32)
    else:
        rt, rh = _i32(rows[0]), _i32(rows[1])
        n_rows = int(rt.size)
        out = np.zeros((n_rows, dv), dtype=np.float64)
    rc = lib.oracle_diffattn_rows(int(cu.size - 1), _ip(cu), H, Hkv, d, dv, _dp(qa), _dp(ka), _dp(va),
                                  _dp(lam_h), float(lam_init), _dp(wa), float(eps), int(bool(causal)),
                                  n_rows, _ip(rt), _ip(rh), _dp(out))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def forward(inp, rows=None, lambda_override=None, lambda_init_override=None) -> np.ndarray:
    """Oracle output for a `workloads.Inputs`: lambda from its vectors, lambda_init
    from its depth, unless overridden."""
    wl = inp.wl
    li = lambda_init(wl.depth) if lambda_init_override is None else float(lambda_init_override)
    lam = (lambda_values(inp.lambda_q1, inp.lambda_k1, inp.lambda_q2, inp.lambda_k2, li)
           if lambda_override is None else lambda_override)
    return forward_rows(inp.cu_seqlens, inp.q, inp.k, inp.v, lam, li, inp.subln_w, wl.eps,
                        wl.causal, rows)


def forward_map_form(cu_seqlens, q, k, v, lam, lam_init: float, w, eps: float,
                     causal: bool) -> np.ndarray:
    """NumPy fp64 brute force in the map-difference form, for small inputs:
    per sequence and head, build A_c = s Q_c K_c^T plus the causal mask of -inf
    above the diagonal, softmax each row, form (A_1 - lambda A_2) and multiply by
    V, then RMSNorm over dv, times w and (1 - lambda_init)."""
    cu = _i32(cu_seqlens)
    qa, ka, va, wa = _f64(q), _f64(k), _f64(v), _f64(w)
    tokens, H, two_d = qa.shape
    Hkv, dv = ka.shape[1], va.shape[2]
    d = two_d // 2
    lam_h = _per_head_lambda(lam, H)
    n_rep = H // Hkv
    s = d ** -0.5
    out = np.zeros((tokens, H, dv), dtype=np.float64)
    for si in range(cu.size - 1):
        a, b = int(cu[si]), int(cu[si + 1])
        n = b - a
        if n == 0:
            continue
        mask = np.zeros((n, n))
        if causal:
            mask[np.triu_indices(n, 1)] = -np.inf
        for h in range(H):
            g = h // n_rep
            maps = []
            for c in range(2):
                qc = qa[a:b, h, c * d:(c + 1) * d]
                kc = ka[a:b, g, c * d:(c + 1) * d]
                A = qc @ kc.T * s + mask
                A = np.exp(A - A.max(axis=1, keepdims=True))
                maps.append(A / A.sum(axis=1, keepdims=True))
            attn = maps[0] - lam_h[h] * maps[1]
            O = attn @ va[a:b, g, :]
            rms = np.sqrt(np.mean(O ** 2, axis=-1, keepdims=True) + eps)
            out[a:b, h, :] = O / rms * wa * (1.0 - lam_init)
    return out
