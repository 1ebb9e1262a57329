"""GB300-native exact multi-head scaled dot-product attention.

Thin Python binding over the C ABI in include/attn.h (libattn_gb300.so, built for sm_103a by
``self_attention_gb300.build``).  This module only marshals arguments: every step of the
computation runs in the library's CUDA kernels.  PyTorch supplies device memory and the
current stream.  If the library is missing or cannot be loaded, every call raises: there is
no fallback implementation.

Operation ("Self-attention, CUDA kernels and FlashAttention", section 1):
    O = softmax(scale * Q K^T) V,  scale = 1/sqrt(d_k) by default,
per (batch, head), with tensors laid out [B, H, N, d_k] bf16.  The forward also returns
LSE = log sum_j exp(scale * q_i . k_j) per row ([B, H, N] fp32), the statistic the backward
pass recomputes the attention tiles from (section 3, "Recomputation in backpropagation").
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from .build import LIB_PATH

__all__ = [
    "AttnError", "attn_fwd", "attn_fwd_workspace_size", "attn_fwd_with_workspace", "attn_fwd_diagnostic",
    "attn_bwd", "attn_bwd_workspace_size", "attn_bwd_preprocess",
    "attn_bwd_main", "attn_bwd_dq_convert", "attn_get_device_status",
    "attn_status_string", "attn_last_error_string", "attn_debug_wait_timeout", "attn_bwd_noalloc",
    "vector_add", "attn_bwd_deterministic", "attn_qkv_proj", "attn_qkv_proj_bwd", "qkv_proj",
    "qkv_proj_backward",
    "forward", "forward_diagnostic", "backward", "attention",
    "load_library", "STATUS",
]

STATUS = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED_DK",
    3: "ATTN_ERR_MISALIGNED", 4: "ATTN_ERR_LAUNCH", 5: "ATTN_ERR_TIMEOUT",
    6: "ATTN_ERR_WORKSPACE", 7: "ATTN_ERR_DEVICE", 8: "ATTN_ERR_TOO_LARGE",
}
EXPORTS = ("attn_fwd", "attn_fwd_workspace_size", "attn_fwd_with_workspace", "attn_fwd_diagnostic", "attn_bwd", "attn_bwd_workspace_size", "attn_bwd_preprocess",
           "attn_bwd_main", "attn_bwd_dq_convert", "attn_get_device_status", "attn_status_string",
           "attn_last_error_string", "attn_debug_wait_timeout", "attn_bwd_noalloc", "vector_add",
           "attn_bwd_deterministic", "attn_qkv_proj", "attn_qkv_proj_bwd",
           "attn_fwd_unfused", "attn_fwd_unfused_workspace_size")


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {attn_status_string(code)}"
        if code == 4:
            msg += f" [{attn_last_error_string()}]"
        super().__init__(msg)


_lib = None
_VP, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def load_library(path: str = LIB_PATH):
    """Load libattn_gb300.so and declare its signatures (no GPU needed to load it)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libattn_gb300.so not found at {path}: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(path)
    lib.attn_fwd.argtypes = [_VP] * 5 + [_I] * 4 + [_F, _VP]
    lib.attn_fwd_workspace_size.argtypes = [_I] * 4
    lib.attn_fwd_workspace_size.restype = _SZ
    lib.attn_fwd_with_workspace.argtypes = [_VP] * 6 + [_SZ] + [_I] * 4 + [_F, _VP]
    lib.attn_fwd_with_workspace.restype = _I
    lib.attn_fwd_diagnostic.argtypes = [_VP] * 6 + [_I] * 4 + [_F, _VP]
    lib.attn_fwd_diagnostic.restype = _I
    lib.attn_fwd.restype = _I
    lib.attn_bwd_workspace_size.argtypes = [_I] * 4
    lib.attn_bwd_workspace_size.restype = _SZ
    lib.attn_bwd.argtypes = [_VP] * 10 + [_SZ] + [_I] * 4 + [_F, _VP]
    lib.attn_bwd.restype = _I
    lib.attn_bwd_preprocess.argtypes = [_VP] * 4 + [_SZ] + [_I] * 4 + [_VP]
    lib.attn_bwd_preprocess.restype = _I
    lib.attn_bwd_main.argtypes = [_VP] * 7 + [_SZ] + [_I] * 4 + [_F, _VP]
    lib.attn_bwd_main.restype = _I
    lib.attn_bwd_dq_convert.argtypes = [_VP, _SZ, _VP] + [_I] * 4 + [_F, _VP]
    lib.attn_bwd_dq_convert.restype = _I
    lib.attn_get_device_status.argtypes = [_VP]
    lib.attn_get_device_status.restype = _I
    lib.attn_status_string.argtypes = [_I]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_last_error_string.argtypes = []
    lib.attn_last_error_string.restype = ctypes.c_char_p
    lib.attn_bwd_deterministic.argtypes = [_VP] * 10 + [_SZ] + [_I] * 4 + [_F, _VP]
    lib.attn_bwd_deterministic.restype = _I
    lib.attn_qkv_proj.argtypes = [_VP] * 7 + [_I] * 5 + [_VP]
    lib.attn_qkv_proj.restype = _I
    lib.attn_qkv_proj_bwd.argtypes = [_VP] * 11 + [_I] * 5 + [_VP]
    lib.attn_qkv_proj_bwd.restype = _I
    lib.vector_add.argtypes = [_VP, _VP, _VP, ctypes.c_longlong, _VP]
    lib.vector_add.restype = _I
    lib.attn_bwd_noalloc.argtypes = [_VP] * 9 + [_I] * 4 + [_F, _VP]
    lib.attn_bwd_noalloc.restype = _I
    lib.attn_fwd_unfused_workspace_size.argtypes = [_I] * 4
    lib.attn_fwd_unfused_workspace_size.restype = _SZ
    lib.attn_fwd_unfused.argtypes = [_VP] * 6 + [_SZ] + [_I] * 4 + [_F, _VP]
    lib.attn_fwd_unfused.restype = _I
    lib.attn_debug_wait_timeout.argtypes = [ctypes.c_uint, _VP]
    lib.attn_debug_wait_timeout.restype = _I
    if path == LIB_PATH:
        _lib = lib
    return lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int:
    return t.data_ptr() if isinstance(t, torch.Tensor) else int(t)


def _raise(code: int, where: str):
    if code != 0:
        raise AttnError(code, where)


def attn_status_string(code: int) -> str:
    try:
        return load_library().attn_status_string(int(code)).decode()
    except RuntimeError:
        return STATUS.get(int(code), f"unknown status {code}")


def attn_last_error_string() -> str:
    return load_library().attn_last_error_string().decode()


# ---------------------------------------------------------------- C-ABI mirrors (same names)
def attn_fwd(q, k, v, o, lse, B: int, H: int, N: int, d_k: int, scale: float, stream=None):
    """Enqueue the forward pass: o and lse written from q, k, v ([B,H,N,d_k] bf16 device)."""
    _raise(load_library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d_k,
                                   float(scale), _stream(stream)), "attn_fwd")


def attn_fwd_workspace_size(B: int, H: int, N: int, d_k: int) -> int:
    return int(load_library().attn_fwd_workspace_size(B, H, N, d_k))


def attn_fwd_with_workspace(q, k, v, o, lse, workspace, workspace_bytes: int, B: int, H: int, N: int,
                            d_k: int, scale: float, stream=None):
    """Enqueue attn_fwd with a caller workspace for the fp16 copy of V (None where
    attn_fwd_workspace_size is 0): the same o and lse, bitwise."""
    _raise(load_library().attn_fwd_with_workspace(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace) if workspace is not None else None,
        workspace_bytes, B, H, N, d_k, float(scale), _stream(stream)), "attn_fwd_with_workspace")


def attn_fwd_diagnostic(q, k, v, o, lse, o32, B: int, H: int, N: int, d_k: int, scale: float, stream=None):
    """Enqueue attn_fwd that also writes O before its bf16 rounding into o32 ([B,H,N,d_k] fp32)."""
    _raise(load_library().attn_fwd_diagnostic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(o32),
                                              B, H, N, d_k, float(scale), _stream(stream)),
           "attn_fwd_diagnostic")


def attn_fwd_unfused_workspace_size(B: int, H: int, N: int, d_k: int) -> int:
    return int(load_library().attn_fwd_unfused_workspace_size(B, H, N, d_k))


def attn_fwd_unfused(q, k, v, o, lse, workspace, workspace_bytes: int, B: int, H: int, N: int,
                     d_k: int, scale: float, stream=None):
    """Enqueue standard attention (S and P through HBM): same outputs as attn_fwd."""
    _raise(load_library().attn_fwd_unfused(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                           workspace_bytes, B, H, N, d_k, float(scale), _stream(stream)),
           "attn_fwd_unfused")


def attn_bwd_workspace_size(B: int, H: int, N: int, d_k: int) -> int:
    return int(load_library().attn_bwd_workspace_size(B, H, N, d_k))


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes: int, B: int, H: int,
             N: int, d_k: int, scale: float, stream=None):
    """Enqueue the backward pass into dq, dk, dv (workspace: caller-owned device memory)."""
    _raise(load_library().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                   int(workspace_bytes), B, H, N, d_k, float(scale),
                                   _stream(stream)), "attn_bwd")


def attn_bwd_preprocess(o, dout, lse, workspace, workspace_bytes: int, B: int, H: int, N: int,
                        d_k: int, stream=None):
    _raise(load_library().attn_bwd_preprocess(_ptr(o), _ptr(dout), _ptr(lse), _ptr(workspace),
                                              int(workspace_bytes), B, H, N, d_k, _stream(stream)),
           "attn_bwd_preprocess")


def attn_bwd_main(q, k, v, dout, dk, dv, workspace, workspace_bytes: int, B: int, H: int, N: int,
                  d_k: int, scale: float, stream=None):
    _raise(load_library().attn_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dk), _ptr(dv),
                                        _ptr(workspace), int(workspace_bytes), B, H, N, d_k,
                                        float(scale), _stream(stream)), "attn_bwd_main")


def attn_bwd_dq_convert(workspace, workspace_bytes: int, dq, B: int, H: int, N: int, d_k: int,
                        scale: float, stream=None):
    _raise(load_library().attn_bwd_dq_convert(_ptr(workspace), int(workspace_bytes), _ptr(dq), B,
                                              H, N, d_k, float(scale), _stream(stream)),
           "attn_bwd_dq_convert")


def attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B: int, H: int, N: int, d_k: int,
                     scale: float, stream=None):
    """attn_bwd without a workspace: for callers that cannot allocate device memory.  The
    scratch is a fixed 64 MiB array inside the library, shared by every call (order calls on
    one stream; overlapping calls race)."""
    _raise(load_library().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout),
                                           _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d_k,
                                           float(scale), _stream(stream)), "attn_bwd_noalloc")


def vector_add(a, b, c, n: int, stream=None):
    """c = a + b for n fp32 device elements (section 2's vector add; the HBM probe)."""
    _raise(load_library().vector_add(_ptr(a), _ptr(b), _ptr(c), int(n), _stream(stream)),
           "vector_add")


def attn_bwd_deterministic(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes: int,
                           B: int, H: int, N: int, d_k: int, scale: float, stream=None):
    """attn_bwd with dQ computed without atomics: bitwise reproducible dQ, dK, dV."""
    _raise(load_library().attn_bwd_deterministic(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(workspace), int(workspace_bytes), B, H, N, d_k, float(scale), _stream(stream)),
        "attn_bwd_deterministic")


def attn_qkv_proj(x, w_q, w_k, w_v, q, k, v, B: int, N: int, D: int, H: int, d_k: int,
                  stream=None):
    _raise(load_library().attn_qkv_proj(_ptr(x), _ptr(w_q), _ptr(w_k), _ptr(w_v), _ptr(q), _ptr(k),
                                        _ptr(v), B, N, D, H, d_k, _stream(stream)), "attn_qkv_proj")


def attn_qkv_proj_bwd(x, w_q, w_k, w_v, dq, dk, dv, dx, dw_q, dw_k, dw_v, B: int, N: int, D: int,
                      H: int, d_k: int, stream=None):
    _raise(load_library().attn_qkv_proj_bwd(
        _ptr(x), _ptr(w_q), _ptr(w_k), _ptr(w_v), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dx),
        _ptr(dw_q), _ptr(dw_k), _ptr(dw_v), B, N, D, H, d_k, _stream(stream)), "attn_qkv_proj_bwd")


def _scratch(nbytes: int, dev, st):
    """Device scratch for a call enqueued on `st`, freed when the caller drops it: torch's
    caching allocator may hand freed memory to the current stream's next allocation, so a
    launch stream other than the current one is recorded on the tensor."""
    t = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = st if isinstance(st, torch.cuda.Stream) else torch.cuda.ExternalStream(int(st), device=dev)
    if s != torch.cuda.current_stream(dev):
        t.record_stream(s)
    return t


def _device_stream(dev, stream):
    """The stream to launch on for tensors on `dev`: the device's current stream by default; a
    torch stream of another device is refused (the kernels would run on one GPU with tensor
    maps over another's memory)."""
    if stream is None:
        return torch.cuda.current_stream(dev)
    if isinstance(stream, torch.cuda.Stream) and stream.device != dev:
        raise ValueError(f"stream is on {stream.device}, tensors on {dev}")
    return stream


def qkv_proj(x, w_q, w_k, w_v, H: int, stream=None):
    """Q, K, V = X W_Q, X W_K, X W_V split into H heads: x [B,N,D] bf16 -> 3 x [B,H,N,D/H] bf16."""
    B, N, D = x.shape
    with torch.cuda.device(x.device):
        st = _device_stream(x.device, stream)
        outs = [torch.empty((B, H, N, D // H), dtype=torch.bfloat16, device=x.device) for _ in range(3)]
        attn_qkv_proj(x, w_q, w_k, w_v, *outs, B, N, D, H, D // H, st)
    return tuple(outs)


def qkv_proj_backward(x, w_q, w_k, w_v, dq, dk, dv, stream=None):
    """Returns (dx [B,N,D] bf16, dw_q, dw_k, dw_v [D,D] fp32)."""
    B, N, D = x.shape
    H = dq.shape[1]
    with torch.cuda.device(x.device):
        st = _device_stream(x.device, stream)
        dx = torch.empty_like(x)
        dws = [torch.empty((D, D), dtype=torch.float32, device=x.device) for _ in range(3)]
        attn_qkv_proj_bwd(x, w_q, w_k, w_v, dq, dk, dv, dx, *dws, B, N, D, H, D // H, st)
    return (dx, *dws)


def attn_get_device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the device status word (0 = ATTN_OK)."""
    return int(load_library().attn_get_device_status(_stream(stream)))


def attn_debug_wait_timeout(limit_us: int, stream=None):
    _raise(load_library().attn_debug_wait_timeout(int(limit_us), _stream(stream)),
           "attn_debug_wait_timeout")


# ---------------------------------------------------------------- tensor-level convenience
def _check_inputs(*ts):
    q = ts[0]
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d_k] tensors")
    for t in ts:
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v (and o, dO) must be contiguous bf16 CUDA tensors of one shape")
        if t.device != q.device:
            raise ValueError("all tensors must be on the same device")
    return q.shape


def forward(q, k, v, scale: float | None = None, stream=None):
    """Returns (o, lse): o [B,H,N,d_k] bf16, lse [B,H,N] fp32 (natural log).  Runs
    attn_fwd_with_workspace, with the fp16 copy of V it wants at long sequences allocated here."""
    B, H, N, D = _check_inputs(q, k, v)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    with torch.cuda.device(q.device):
        st = _device_stream(q.device, stream)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
        nbytes = attn_fwd_workspace_size(B, H, N, D)
        ws = _scratch(nbytes, q.device, st) if nbytes else None
        attn_fwd_with_workspace(q, k, v, o, lse, ws, nbytes, B, H, N, D, scale, st)
    return o, lse


def forward_diagnostic(q, k, v, scale: float | None = None, stream=None):
    """(o, lse, o32): forward()'s results and O before its bf16 rounding (fp32), for measuring
    the kernel's own error apart from the output rounding."""
    B, H, N, D = _check_inputs(q, k, v)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    with torch.cuda.device(q.device):
        st = _device_stream(q.device, stream)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
        o32 = torch.empty((B, H, N, D), dtype=torch.float32, device=q.device)
        attn_fwd_diagnostic(q, k, v, o, lse, o32, B, H, N, D, scale, st)
    return o, lse, o32


def forward_unfused(q, k, v, scale: float | None = None, stream=None):
    """Standard attention (attn_fwd_unfused): returns (o, lse) like forward(), allocating the
    6 B H N^2 bytes of S and P it materialises."""
    B, H, N, D = _check_inputs(q, k, v)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    with torch.cuda.device(q.device):
        st = _device_stream(q.device, stream)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
        nbytes = attn_fwd_unfused_workspace_size(B, H, N, D)
        ws = _scratch(nbytes, q.device, st)
        attn_fwd_unfused(q, k, v, o, lse, ws, nbytes, B, H, N, D, scale, st)
    return o, lse


def backward(q, k, v, o, dout, lse, scale: float | None = None, stream=None, workspace=None,
             deterministic: bool = False):
    """Returns (dq, dk, dv) bf16 for the loss gradient dout = dL/dO.  deterministic=True uses
    attn_bwd_deterministic (no atomics; bitwise reproducible)."""
    B, H, N, D = _check_inputs(q, k, v, o, dout)
    if lse.device != q.device or (workspace is not None and workspace.device != q.device):
        raise ValueError("lse and the workspace must be on the tensors' device")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    with torch.cuda.device(q.device):
        st = _device_stream(q.device, stream)
        nbytes = attn_bwd_workspace_size(B, H, N, D)
        if workspace is None:
            workspace = _scratch(nbytes, q.device, st)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fn = attn_bwd_deterministic if deterministic else attn_bwd
        fn(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace.numel(), B, H, N, D, scale, st)
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, scale):
        o, lse = forward(q, k, v, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.scale = scale
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = backward(q, k, v, o, dout.contiguous(), lse, ctx.scale)
        return dq, dk, dv, None


def attention(q, k, v, scale: float | None = None):
    """softmax(scale * Q K^T) V with autograd support."""
    D = q.shape[-1]
    return _Attention.apply(q, k, v, 1.0 / math.sqrt(D) if scale is None else scale)
