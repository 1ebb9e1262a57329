"""Oracle for exact multi-head scaled dot-product attention (fp64, CPU).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg are the only callers.  The GPU library (``self_attention_gb300``) never imports
this package and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, the N x N score matrix
materialised per head).  This module compiles it with gcc and marshals numpy arrays.

Source: "Self-attention, CUDA kernels and FlashAttention", section 1 (the "Scores",
softmax and "Attention(Q,K,V)" formulas; independent heads) and section 3 ("Recomputation in
backpropagation": the per-row normalisation statistic, here the natural-log LSE).  The
backward is the chain rule applied to those formulas; the article prints none.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)


def compile_shared(src: str, out: str, extra_flags=()) -> None:
    """gcc -O3 -fopenmp -shared; falls back to a serial build if OpenMP is unavailable."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O3", "-std=c11", "-fPIC", "-shared", *extra_flags, src, "-o", out, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            compile_shared(_SRC, tmp)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    lib = ctypes.CDLL(path)
    i64, dbl = ctypes.c_int64, ctypes.c_double
    lib.oracle_attn_fwd.argtypes = [_D, _D, _D, _D, _D, i64, i64, i64, dbl]
    lib.oracle_attn_bwd.argtypes = [_D] * 11 + [i64, i64, i64, dbl]
    lib.oracle_attn_fwd_rows.argtypes = [_D, _D, _D, _I64, i64, _D, _D, i64, i64, dbl]
    lib.oracle_attn_bwd_rows.argtypes = [_D, _D, _D, _D, _I64, i64, _I64, i64, _D, _D, _D,
                                         i64, i64, dbl]
    for f in (lib.oracle_attn_fwd, lib.oracle_attn_bwd, lib.oracle_attn_fwd_rows,
              lib.oracle_attn_bwd_rows):
        f.restype = ctypes.c_int
    _F = ctypes.POINTER(ctypes.c_float)
    lib.oracle_vector_add.argtypes = [_F, _F, _F, i64]
    lib.oracle_vector_add.restype = None
    return lib


def _get():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: widen exactly (bf16/fp32 -> fp64)
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _check(rc: int):
    if rc != 0:
        raise MemoryError("oracle: out of host memory")


def _shape4(q: np.ndarray):
    if q.ndim != 4:
        raise ValueError("expected [B,H,N,d]")
    b, h, n, d = q.shape
    return b, h, n, d


def fwd(q, k, v, scale: float, lib=None):
    """O = softmax(scale * Q K^T) V and LSE, for [B,H,N,d] inputs.  Returns (o, lse) fp64."""
    lib = lib or _get()
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, h, n, d = _shape4(q)
    o = np.empty_like(q)
    lse = np.empty((b, h, n), np.float64)
    _check(lib.oracle_attn_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), b * h, n, d, float(scale)))
    return o, lse


def bwd(q, k, v, dout, scale: float, lib=None):
    """Gradients of <dO, O> with respect to Q, K, V.

    Returns a dict with dq, dk, dv (fp64 [B,H,N,d]), the oracle's own o and lse, D = rowsum(dO o O)
    and Dprime = rowsum(P o dP) ([B,H,N])."""
    lib = lib or _get()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    b, h, n, d = _shape4(q)
    out = {name: np.empty_like(q) for name in ("dq", "dk", "dv", "o")}
    for name in ("lse", "D", "Dprime"):
        out[name] = np.empty((b, h, n), np.float64)
    _check(lib.oracle_attn_bwd(_p(q), _p(k), _p(v), _p(dout), _p(out["dq"]), _p(out["dk"]),
                               _p(out["dv"]), _p(out["o"]), _p(out["lse"]), _p(out["D"]),
                               _p(out["Dprime"]), b * h, n, d, float(scale)))
    return out


def fwd_rows(q_head, k_head, v_head, rows, scale: float, lib=None):
    """Forward for the listed query rows of one head ([N,d] inputs).  Returns (o_rows, lse_rows)."""
    lib = lib or _get()
    q, k, v = _f64(q_head), _f64(k_head), _f64(v_head)
    n, d = q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= n):
        raise IndexError("row index out of range")
    o = np.empty((rows.size, d), np.float64)
    lse = np.empty(rows.size, np.float64)
    _check(lib.oracle_attn_fwd_rows(_p(q), _p(k), _p(v), rows.ctypes.data_as(_I64), rows.size,
                                    _p(o), _p(lse), n, d, float(scale)))
    return o, lse


def bwd_rows(q_head, k_head, v_head, do_head, qrows, krows, scale: float, lib=None):
    """dQ for query rows ``qrows`` and dK, dV for key rows ``krows`` of one head ([N,d] inputs)."""
    lib = lib or _get()
    q, k, v, dout = _f64(q_head), _f64(k_head), _f64(v_head), _f64(do_head)
    n, d = q.shape
    qrows = np.ascontiguousarray(qrows, dtype=np.int64)
    krows = np.ascontiguousarray(krows, dtype=np.int64)
    for r in (qrows, krows):
        if r.size and (r.min() < 0 or r.max() >= n):
            raise IndexError("row index out of range")
    dq = np.empty((qrows.size, d), np.float64)
    dk = np.empty((krows.size, d), np.float64)
    dv = np.empty((krows.size, d), np.float64)
    _check(lib.oracle_attn_bwd_rows(_p(q), _p(k), _p(v), _p(dout), qrows.ctypes.data_as(_I64),
                                    qrows.size, krows.ctypes.data_as(_I64), krows.size, _p(dq),
                                    _p(dk), _p(dv), n, d, float(scale)))
    return dq, dk, dv


def vector_add(a, b, lib=None):
    """c = a + b element-wise in fp32 (section 2's vector add).  Returns a new float32 array."""
    lib = lib or _get()
    a = np.ascontiguousarray(a, dtype=np.float32).ravel()
    b = np.ascontiguousarray(b, dtype=np.float32).ravel()
    if a.size != b.size:
        raise ValueError("a and b differ in length")
    c = np.empty_like(a)
    fp = ctypes.POINTER(ctypes.c_float)
    lib.oracle_vector_add(a.ctypes.data_as(fp), b.ctypes.data_as(fp), c.ctypes.data_as(fp), a.size)
    return c


# ---------------------------------------------------------------- QKV projection
# "Self-attention, CUDA kernels and FlashAttention", section 1 ("Generating queries, keys and
# values"): Q = X W_Q, K = X W_K, V = X W_V, with W in R^(D x d_k) per head; the heads' weights
# side by side form one D x D matrix, head h taking columns [h*d_k, (h+1)*d_k).  Plain fp64 matrix
# products (numpy) followed by the split of the columns into heads.

def _heads(y, H):
    """[B, N, D] -> [B, H, N, D/H]: head h = columns [h*d, (h+1)*d)."""
    B, N, D = y.shape
    return np.ascontiguousarray(y.reshape(B, N, H, D // H).transpose(0, 2, 1, 3))


def _merge(z):
    """[B, H, N, d] -> [B, N, H*d], the inverse of _heads."""
    B, H, N, d = z.shape
    return np.ascontiguousarray(z.transpose(0, 2, 1, 3).reshape(B, N, H * d))


def qkv_proj(x, w_q, w_k, w_v, H):
    """x [B, N, D]; w_* [D, D].  Returns (q, k, v), each [B, H, N, D/H] fp64."""
    x = _f64(x)
    return tuple(_heads(x @ _f64(w), H) for w in (w_q, w_k, w_v))


def qkv_proj_bwd(x, w_q, w_k, w_v, dq, dk, dv):
    """Gradients of sum_t <dY_t, Y_t> for Y_t = X W_t (heads merged back into columns):
    dX = sum_t dY_t W_t^T and dW_t = X^T dY_t (summed over the batch).  Returns
    (dx [B,N,D], dw_q, dw_k, dw_v [D,D]) in fp64."""
    x = _f64(x)
    B, N, D = x.shape
    xf = x.reshape(B * N, D)
    dx = np.zeros((B * N, D))
    dws = []
    for w, dy in ((w_q, dq), (w_k, dk), (w_v, dv)):
        g = _merge(_f64(dy)).reshape(B * N, D)
        dx += g @ _f64(w).T
        dws.append(xf.T @ g)
    return (dx.reshape(B, N, D), *dws)
