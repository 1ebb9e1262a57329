"""The C-ABI calls enqueue only on the stream they are given and never synchronise, so a whole
forward + backward step can be captured once in a CUDA graph and replayed: replays with new
inputs copied into the captured buffers must give what eager calls give."""
import math

import numpy as np
import pytest
import torch

import self_attention_gb300 as sa
from self_attention_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_attention_gb300.build import build
    sa.load_library(build())


@pytest.mark.parametrize("shape", [(4, 12, 196, 64), (1, 4, 1000, 128), (1, 96, 200, 64)])
def test_graph_replay_matches_eager(shape):
    """The last shape takes the whole-head backward (d_k = 64, N <= 256, one head per CTA)."""
    B, H, N, D = shape
    scale = 1.0 / math.sqrt(D)
    dev = lambda t: t.cuda()
    bufs = {x: torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda") for x in ("q", "k", "v", "do")}
    o, dq, dk, dv = (torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    lse = torch.empty(B, H, N, device="cuda")
    wsb = sa.attn_bwd_workspace_size(B, H, N, D)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def step():
        sa.attn_fwd(bufs["q"], bufs["k"], bufs["v"], o, lse, B, H, N, D, scale, s)
        sa.attn_bwd(bufs["q"], bufs["k"], bufs["v"], o, bufs["do"], lse, dq, dk, dv, ws, wsb, B, H, N,
                    D, scale, s)

    first = make_qkv(B, H, N, D, seed=9100 + N, with_do=True)
    for x in bufs:
        bufs[x].copy_(first[x])
    torch.cuda.synchronize()
    with torch.cuda.stream(s):   # warm-up outside the capture (loads the kernels)
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    torch.cuda.synchronize()

    for seed in (9200 + N, 9300 + N):
        inp = make_qkv(B, H, N, D, seed=seed, with_do=True)
        for x in bufs:
            bufs[x].copy_(inp[x])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert sa.attn_get_device_status() == 0
        replay = {n_: t.float().cpu().numpy() for n_, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
        ref_o, ref_lse = sa.forward(*(dev(inp[x]) for x in ("q", "k", "v")), scale)
        ref_dq, ref_dk, ref_dv = sa.backward(*(dev(inp[x]) for x in ("q", "k", "v")), ref_o, dev(inp["do"]),
                                             ref_lse, scale)
        eager = {n_: t.float().cpu().numpy() for n_, t in (("o", ref_o), ("lse", ref_lse), ("dq", ref_dq), ("dk", ref_dk), ("dv", ref_dv))}
        # forward, dK and dV involve no atomics: bitwise equal; dQ sums fp32 partials in any order
        for n_ in ("o", "lse", "dk", "dv"):
            np.testing.assert_array_equal(replay[n_], eager[n_], err_msg=n_)
        np.testing.assert_allclose(replay["dq"], eager["dq"], rtol=2 ** -7, atol=2 ** -12)


@pytest.mark.parametrize("shape", [(8, 12, 196, 64), (1, 4, 700, 128)])
def test_graph_replay_deterministic_bitwise(shape):
    """The deterministic backward has no atomics: a replayed graph of forward + deterministic
    backward reproduces eager calls bit for bit, dQ included."""
    B, H, N, D = shape
    scale = 1.0 / math.sqrt(D)
    bufs = {x: torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda") for x in ("q", "k", "v", "do")}
    o, dq, dk, dv = (torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    lse = torch.empty(B, H, N, device="cuda")
    wsb = sa.attn_bwd_workspace_size(B, H, N, D)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def step(outs):
        o_, lse_, dq_, dk_, dv_ = outs
        sa.attn_fwd(bufs["q"], bufs["k"], bufs["v"], o_, lse_, B, H, N, D, scale, s)
        sa.attn_bwd_deterministic(bufs["q"], bufs["k"], bufs["v"], o_, bufs["do"], lse_, dq_, dk_, dv_,
                                  ws, wsb, B, H, N, D, scale, s)

    outs = (o, lse, dq, dk, dv)
    first = make_qkv(B, H, N, D, seed=9400 + N, with_do=True)
    for x in bufs:
        bufs[x].copy_(first[x])
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step(outs)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(outs)
    torch.cuda.synchronize()
    inp = make_qkv(B, H, N, D, seed=9500 + N, with_do=True)
    for x in bufs:
        bufs[x].copy_(inp[x])
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert sa.attn_get_device_status() == 0
    replay = [t.float().cpu().numpy() for t in outs]
    eager_outs = tuple(torch.empty_like(t) for t in outs)
    with torch.cuda.stream(s):
        step(eager_outs)
    torch.cuda.synchronize()
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), replay, (t.float().cpu().numpy() for t in eager_outs)):
        np.testing.assert_array_equal(a, b, err_msg=name)


@pytest.mark.parametrize("shape", [(1, 4, 2048, 64), (1, 2, 8192, 128)])
def test_graph_replay_forward_with_workspace(shape):
    """attn_fwd_with_workspace (V rounded to fp16 into the workspace, then the forward kernel)
    captured once with fixed buffers and replayed on new inputs: O and LSE equal eager forward()
    bit for bit."""
    B, H, N, D = shape
    scale = 1.0 / math.sqrt(D)
    fwsb = sa.attn_fwd_workspace_size(B, H, N, D)
    assert fwsb > 0
    fws = torch.empty(fwsb, dtype=torch.uint8, device="cuda")
    bufs = {x: torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda") for x in ("q", "k", "v")}
    o = torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, N, device="cuda")
    s = torch.cuda.Stream()

    def step():
        sa.attn_fwd_with_workspace(bufs["q"], bufs["k"], bufs["v"], o, lse, fws, fwsb, B, H, N, D, scale, s)

    first = make_qkv(B, H, N, D, seed=9600 + N, with_do=False)
    for x in bufs:
        bufs[x].copy_(first[x])
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    torch.cuda.synchronize()
    for seed in (9700 + N, 9800 + N):
        inp = make_qkv(B, H, N, D, seed=seed, with_do=False)
        for x in bufs:
            bufs[x].copy_(inp[x])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert sa.attn_get_device_status() == 0
        ref_o, ref_lse = sa.forward(*(inp[x].cuda() for x in ("q", "k", "v")), scale)
        assert torch.equal(o, ref_o)
        assert torch.equal(lse, ref_lse)
