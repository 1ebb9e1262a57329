"""The QKV projection (section 1: Q = X W_Q, K = X W_K, V = X W_V, one d_k-wide column block
per head) and its backward on the GPU, through the C ABI, against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import self_attention_gb300 as sa
from self_attention_gb300.inputs import WORKLOADS, make_block_inputs
from _compare import check_grad, rel_fro

pytestmark = pytest.mark.gpu

PROJ_REL = 1e-2   # bf16 outputs of fp32 sums: relative Frobenius bound for Q, K, V and dX
DW_REL = 1e-4     # fp32 dW from exact bf16 products summed in fp32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_attention_gb300.build import build
    sa.load_library(build())


def _draw(B, N, D, H, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, N, D, generator=g).bfloat16()
    ws = [(torch.randn(D, D, generator=g) / math.sqrt(D)).bfloat16() for _ in range(3)]
    dys = [torch.randn(B, H, N, D // H, generator=g).bfloat16() for _ in range(3)]
    return x, ws, dys


SHAPES = [(2, 130, 256, 4), (1, 77, 256, 2), (3, 64, 384, 6), (1, 200, 512, 4)]


@pytest.mark.parametrize("B,N,D,H", SHAPES)
def test_proj_forward_and_backward(B, N, D, H):
    x, ws, dys = _draw(B, N, D, H, seed=B * 1000 + N + D)
    xc, wc, dyc = x.cuda(), [w.cuda() for w in ws], [d.cuda() for d in dys]
    q, k, v = sa.qkv_proj(xc, *wc, H)
    dx, dwq, dwk, dwv = sa.qkv_proj_backward(xc, *wc, *dyc)
    assert sa.attn_get_device_status() == 0
    ref = oracle.qkv_proj(x, *ws, H)
    for name, got, r in zip("qkv", (q, k, v), ref):
        rf = rel_fro(got.float().cpu().numpy(), r)
        assert rf <= PROJ_REL, f"{name}: relative Frobenius {rf:.3g}"
    rdx, *rdw = oracle.qkv_proj_bwd(x, *ws, *dys)
    check_grad("dx", dx.float().cpu().numpy(), rdx, f"{B},{N},{D},{H}")
    for name, got, r in zip(("dw_q", "dw_k", "dw_v"), (dwq, dwk, dwv), rdw):
        rf = rel_fro(got.cpu().numpy(), r)
        assert rf <= DW_REL, f"{name}: relative Frobenius {rf:.3g}"


def test_proj_matches_block_input_preparation():
    """On the full ViT-B block workload (X 32 x 576 x 768, 12 heads), the GPU projection agrees
    with the fp32 CPU projection the workload's inputs are made with to one bf16 spacing (both
    round an fp32 sum of 768 products, summed in different orders: a spacing, plus 1e-5 for the
    fp32 summation error near zero, where the spacing itself is tiny), and with the fp64 oracle
    in relative Frobenius norm."""
    w = WORKLOADS["vit_b_mhsa_block"]
    inp = make_block_inputs(w)
    q, k, v = sa.qkv_proj(inp["x"].cuda(), inp["w_q"].cuda(), inp["w_k"].cuda(), inp["w_v"].cuda(), w.H)
    ref = oracle.qkv_proj(inp["x"], inp["w_q"], inp["w_k"], inp["w_v"], w.H)
    for name, got, cpu, r in zip("qkv", (q, k, v), (inp["q"], inp["k"], inp["v"]), ref):
        g, c = got.float().cpu(), cpu.float()
        big = torch.maximum(g.abs(), c.abs()).clamp_min(2 ** -100)
        spacing = 2.0 ** (torch.floor(torch.log2(big)) - 7)
        bad = (g - c).abs() > spacing + 1e-5
        assert not bool(bad.any()), f"{name}: {int(bad.sum())} elements beyond one bf16 spacing"
        assert rel_fro(g.numpy(), r) <= PROJ_REL


def test_block_forward_backward_end_to_end():
    """Projection -> attention forward -> attention backward -> projection backward, all on the
    GPU, against the same chain of fp64 oracle functions."""
    B, N, D, H = 2, 130, 256, 4
    x, ws, _ = _draw(B, N, D, H, seed=77)
    g = torch.Generator().manual_seed(78)
    do = torch.randn(B, H, N, D // H, generator=g).bfloat16()
    xc, wc = x.cuda(), [w.cuda() for w in ws]
    q, k, v = sa.qkv_proj(xc, *wc, H)
    o, lse = sa.forward(q, k, v)
    dq, dk, dv = sa.backward(q, k, v, o, do.cuda(), lse)
    dx, dwq, dwk, dwv = sa.qkv_proj_backward(xc, *wc, dq, dk, dv)
    assert sa.attn_get_device_status() == 0
    rq, rk, rv = oracle.qkv_proj(x, *ws, H)
    scale = 1.0 / math.sqrt(D // H)
    rg = oracle.bwd(rq, rk, rv, do, scale)
    rdx, *rdw = oracle.qkv_proj_bwd(x, *ws, rg["dq"], rg["dk"], rg["dv"])
    check_grad("dx", dx.float().cpu().numpy(), rdx, "block")
    for name, got, r in zip(("dw_q", "dw_k", "dw_v"), (dwq, dwk, dwv), rdw):
        check_grad(name, got.cpu().numpy(), r, "block")


def test_proj_argument_errors():
    x, ws, _ = _draw(1, 8, 256, 4, seed=5)
    xc, wc = x.cuda(), [w.cuda() for w in ws]
    out = [torch.empty(1, 4, 8, 64, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    with pytest.raises(sa.AttnError) as e:          # D != H * d_k
        sa.attn_qkv_proj(xc, *wc, *out, 1, 8, 256, 3, 64)
    assert e.value.code == 1
    with pytest.raises(sa.AttnError) as e:
        sa.attn_qkv_proj(xc, *wc, *out, 1, 8, 256, 8, 32)
    assert e.value.code == 2
    with pytest.raises(sa.AttnError) as e:          # output aliasing the input
        sa.attn_qkv_proj(xc, *wc, xc, out[1], out[2], 1, 8, 256, 4, 64)
    assert e.value.code == 1
