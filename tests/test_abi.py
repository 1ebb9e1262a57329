"""The C-ABI library without a GPU: it loads, exports every function include/attn.h declares,
and rejects bad arguments with the documented status before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

import self_attention_gb300 as sa
from self_attention_gb300.build import INCLUDE, build

HEADER = os.path.join(INCLUDE, "attn.h")


@pytest.fixture(scope="module")
def lib():
    return sa.load_library(build())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:attn_status|size_t|const char \*)\s*(\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_get_device_status",
                     "attn_status_string", "vector_add", "attn_bwd_noalloc"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build()], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, f"{name} declared in attn.h but not exported"
        assert hasattr(lib, name)
    assert set(sa.EXPORTS) <= exported


def test_status_strings(lib):
    for code, name in sa.STATUS.items():
        assert sa.attn_status_string(code).startswith(name)


def test_workspace_size(lib):
    a256 = lambda x: (x + 255) // 256 * 256
    assert sa.attn_bwd_workspace_size(1, 1, 100, 64) == 2 * a256(128 * 4) + a256(100 * 64 * 4)
    assert (sa.attn_bwd_workspace_size(2, 16, 16384, 128)
            == 2 * a256(32 * 16384 * 4) + a256(32 * 16384 * 128 * 4))
    assert sa.attn_bwd_workspace_size(1, 1, 100, 96) == 0
    assert sa.attn_bwd_workspace_size(0, 1, 100, 64) == 0


# Fake, never-dereferenced device addresses: validation fails before any CUDA call.
Q, K, V, O, L = (0x10000000 * (i + 1) for i in range(5))


def _fwd(lib, q=Q, k=K, v=V, o=O, lse=L, B=1, H=2, N=64, d=64, scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), None)


def test_fwd_argument_errors(lib):
    assert _fwd(lib, d=96) == 2
    assert _fwd(lib, d=0) == 2
    assert _fwd(lib, B=0) == 1
    assert _fwd(lib, N=0) == 1
    assert _fwd(lib, H=-1) == 1
    assert _fwd(lib, scale=float("nan")) == 1
    assert _fwd(lib, scale=0.0) == 1
    assert _fwd(lib, scale=float("inf")) == 1
    assert _fwd(lib, q=0) == 1
    assert _fwd(lib, lse=0) == 1
    assert _fwd(lib, q=Q + 8) == 3
    assert _fwd(lib, lse=L + 4) == 3
    assert _fwd(lib, o=Q) == 1                 # output aliases an input
    assert _fwd(lib, lse=O + 64) == 1          # lse inside o
    assert _fwd(lib, B=1 << 20, H=1 << 20) == 1


def test_fwd_workspace_size_and_argument_errors(lib):
    a256 = lambda x: (x + 255) // 256 * 256
    # an fp16 copy of V from N = 2048 (d_k = 64) and N = 8192 (d_k = 128) on, none below
    assert sa.attn_fwd_workspace_size(1, 2, 2047, 64) == 0
    assert sa.attn_fwd_workspace_size(1, 2, 8191, 128) == 0
    assert sa.attn_fwd_workspace_size(1, 2, 2048, 64) == a256(2 * 2048 * 64 * 2)
    assert sa.attn_fwd_workspace_size(2, 16, 16384, 128) == 32 * 16384 * 128 * 2
    assert sa.attn_fwd_workspace_size(1, 2, 4096, 96) == 0
    assert sa.attn_fwd_workspace_size(0, 2, 4096, 64) == 0
    need = sa.attn_fwd_workspace_size(1, 2, 2048, 64)
    ws = 0x70000000

    def fwd(ws=ws, nbytes=need, N=2048, d=64, o=O):
        return lib.attn_fwd_with_workspace(Q, K, V, o, L, ws, nbytes, 1, 2, N, d, ctypes.c_float(0.125), None)

    assert fwd(d=96) == 2
    assert fwd(ws=0) == 6
    assert fwd(nbytes=need - 1) == 6
    assert fwd(ws=ws + 16) == 6
    assert fwd(ws=V) == 1                 # the fp16 copy over an input
    assert fwd(ws=O + 256) == 1           # ... over the output
    assert fwd(o=Q) == 1
    # below the threshold the call is attn_fwd: no workspace needed, the same checks
    assert fwd(ws=0, nbytes=0, N=64, o=Q) == 1
    assert fwd(ws=0, nbytes=0, N=64, d=128, o=Q + 8) == 3


def test_fwd_diagnostic_argument_errors(lib):
    o32 = 0x70000000

    def fwd(o32=o32, o=O, d=64):
        return lib.attn_fwd_diagnostic(Q, K, V, o, L, o32, 1, 2, 64, d, ctypes.c_float(0.125), None)

    assert fwd(d=96) == 2
    assert fwd(o32=0) == 1
    assert fwd(o32=o32 + 4) == 3
    assert fwd(o32=Q) == 1                # over an input
    assert fwd(o32=O + 64) == 1           # over the bf16 output
    assert fwd(o=Q) == 1


def test_bwd_argument_errors(lib):
    ws = 0x70000000
    need = sa.attn_bwd_workspace_size(1, 2, 64, 64)
    dq, dk, dv = 0x80000000, 0x90000000, 0xA0000000

    def bwd(ws=ws, nbytes=need, d=64, dq=dq, o=O):
        return lib.attn_bwd(Q, K, V, o, 0x60000000, L, dq, dk, dv, ws, nbytes, 1, 2, 64, d,
                            ctypes.c_float(0.125), None)

    assert bwd(d=80) == 2
    assert bwd(nbytes=need - 1) == 6
    assert bwd(ws=0) == 6
    assert bwd(ws=ws + 16) == 6
    assert bwd(dq=Q) == 1
    assert bwd(dq=dk) == 1
    assert bwd(dq=dq + 2) == 3
    assert bwd(o=0) == 1
    assert lib.attn_bwd_main(Q, K, V, 0x60000000, dk, dv, ws, need - 16, 1, 2, 64, 64,
                             ctypes.c_float(0.125), None) == 6
    assert lib.attn_bwd_preprocess(O, 0, L, ws, need, 1, 2, 64, 64, None) == 1
    assert lib.attn_bwd_preprocess(O, 0x60000000, 0, ws, need, 1, 2, 64, 64, None) == 1
    assert lib.attn_bwd_dq_convert(ws, need, 0, 1, 2, 64, 64, ctypes.c_float(0.125), None) == 1


def test_unfused_workspace_and_argument_errors(lib):
    a256 = lambda x: (x + 255) // 256 * 256
    assert sa.attn_fwd_unfused_workspace_size(1, 2, 100, 64) == a256(2 * 100 * 100 * 4) + a256(2 * 100 * 100 * 2)
    assert sa.attn_fwd_unfused_workspace_size(1, 2, 100, 96) == 0
    assert sa.attn_fwd_unfused_workspace_size(1, 1 << 16, 1 << 16, 64) == 0   # B*H*N^2 >= 2^40
    ws = 0x70000000
    need = sa.attn_fwd_unfused_workspace_size(1, 2, 64, 64)

    def unf(ws=ws, nbytes=need, d=64, o=O, q=Q, lse=L):
        return lib.attn_fwd_unfused(q, K, V, o, lse, ws, nbytes, 1, 2, 64, d, ctypes.c_float(0.125), None)

    assert unf(d=80) == 2
    assert unf(nbytes=need - 1) == 6
    assert unf(ws=0) == 6
    assert unf(ws=ws + 16) == 6
    assert unf(q=0) == 1
    assert unf(q=Q + 8) == 3
    assert unf(o=Q) == 1                       # output over an input
    assert unf(o=ws + 256) == 1                # output inside the workspace
    assert unf(lse=O + 64) == 1                # lse inside o


def test_debug_timeout_argument_range(lib):
    assert lib.attn_debug_wait_timeout(0, None) == 1
    assert lib.attn_debug_wait_timeout(10 ** 7, None) == 1


def test_vector_add_argument_errors(lib):
    assert lib.vector_add(Q, K, V, -1, None) == 1
    assert lib.vector_add(Q, K, V, 0, None) == 0          # nothing to do
    assert lib.vector_add(0, K, V, 16, None) == 1
    assert lib.vector_add(Q + 4, K, V, 16, None) == 3
    assert lib.vector_add(Q, K, Q + 16, 16, None) == 1    # partial overlap with an input


def test_noalloc_and_deterministic_argument_errors(lib):
    """attn_bwd_noalloc checks the sizes and its fixed 64 MiB scratch, and
    attn_bwd_deterministic the same arguments as attn_bwd, before either touches the device."""
    z = [0] * 9
    assert lib.attn_bwd_workspace_size(2, 16, 16384, 128) > 64 << 20
    assert lib.attn_bwd_noalloc(*z, 2, 16, 16384, 128, ctypes.c_float(0.088), None) == 8
    assert lib.attn_bwd_noalloc(*z, 1, 2, 64, 80, ctypes.c_float(0.125), None) == 2
    assert lib.attn_bwd_noalloc(*z, 0, 2, 64, 64, ctypes.c_float(0.125), None) == 1
    assert lib.attn_bwd_noalloc(*z, 1, 2, 64, 64, ctypes.c_float(float("nan")), None) == 1

    ws = 0x70000000
    need = sa.attn_bwd_workspace_size(1, 2, 64, 64)
    dq, dk, dv = 0x80000000, 0x90000000, 0xA0000000

    def det(ws=ws, nbytes=need, d=64, dq=dq, dk=dk):
        return lib.attn_bwd_deterministic(Q, K, V, O, 0x60000000, L, dq, dk, dv, ws, nbytes, 1, 2, 64,
                                          d, ctypes.c_float(0.125), None)

    assert det(d=96) == 2
    assert det(nbytes=need - 1) == 6
    assert det(ws=ws + 64) == 6
    assert det(dq=K) == 1            # an output aliasing an input
    assert det(dk=dq) == 1           # two outputs overlapping
    assert det(dq=dq + 8) == 3


def test_qkv_proj_argument_errors(lib):
    """The projection calls check sizes, pointers, alignment and overlaps before the device."""
    X = 0x10000000                                   # [1, 8, 256] bf16: 4 KB
    W = (0x20000000, 0x21000000, 0x22000000)         # [256, 256] bf16: 128 KB each
    OUT = (0x30000000, 0x31000000, 0x32000000)

    def fwd(B=1, N=8, D=256, H=4, d=64, x=X, w=W, o=OUT):
        return lib.attn_qkv_proj(x, *w, *o, B, N, D, H, d, None)

    assert fwd(d=32) == 2
    assert fwd(H=3) == 1                             # D != H * d_k
    assert fwd(D=192, H=3) == 1                      # D not a multiple of 128
    assert fwd(B=0) == 1
    assert fwd(x=0) == 1
    assert fwd(w=(W[0], 0, W[2])) == 1
    assert fwd(x=X + 8) == 3
    assert fwd(o=(OUT[0], 0, OUT[2])) == 1
    assert fwd(o=(OUT[0] + 2, OUT[1], OUT[2])) == 3
    assert fwd(o=(X, OUT[1], OUT[2])) == 1           # an output over the input
    assert fwd(o=(OUT[0], W[1], OUT[2])) == 1        # an output over a weight
    assert fwd(o=(OUT[0], OUT[0] + 16, OUT[2])) == 1  # two outputs overlapping
    # B * N token rows past the int range, though B * N * D stays under the 2^40 element bound
    assert fwd(B=2, N=1 << 30, D=128, H=2) == 1
    assert lib.attn_qkv_proj_bwd(X, *W, 0x60000000, 0x61000000, 0x62000000, 0x40000000,
                                 0x50000000, 0x51000000, 0x52000000, 2, 1 << 30, 128, 2, 64, None) == 1

    DY = (0x60000000, 0x61000000, 0x62000000)
    DW = (0x50000000, 0x51000000, 0x52000000)        # [256, 256] fp32: 256 KB each

    def bwd(dx=0x40000000, dw=DW, dy=DY, d=64):
        return lib.attn_qkv_proj_bwd(X, *W, *dy, dx, *dw, 1, 8, 256, 4, d, None)

    assert bwd(d=96) == 2
    assert bwd(dx=0) == 1
    assert bwd(dx=0x40000008) == 3
    assert bwd(dy=(DY[0], DY[1], 0)) == 1
    assert bwd(dw=(DW[0], 0, DW[2])) == 1
    assert bwd(dw=(DW[0] + 4, DW[1], DW[2])) == 3
    assert bwd(dx=X) == 1                            # dX over X
    assert bwd(dw=(DY[1], DW[1], DW[2])) == 1        # a dW over an incoming gradient
    assert bwd(dw=(DW[0], DW[0] + 1024, DW[2])) == 1  # two dW overlapping
