"""Backward parity: dQ, dK, dV from the CUDA path (through the C ABI) against the fp64 oracle
on the same seeded bf16 inputs.  The GPU backward consumes the GPU forward's bf16 O and
fp32 LSE, exactly as a training step does; the oracle uses its own fp64 forward."""
import math

import numpy as np
import pytest
import torch

import oracle
import self_attention_gb300 as sa
from self_attention_gb300.inputs import WORKLOADS, make_qkv, make_workload_inputs
from _compare import GRAD_REL_FRO, check_grad, rel_fro

pytestmark = pytest.mark.gpu

GUARD = 16384


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_attention_gb300.build import build
    sa.load_library(build())


def _guarded(shape, dtype):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(shape)


def _intact(buf):
    return bool(torch.isnan(torch.cat([buf[:GUARD], buf[-GUARD:]])).all())


def run_fwd_bwd(inp, scale, deterministic=False):
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    B, H, N, D = q.shape
    o, lse = sa.forward(q, k, v, scale)
    bufs = [_guarded((B, H, N, D), torch.bfloat16) for _ in range(3)]
    dq, dk, dv = (b[1] for b in bufs)
    ws_bytes = sa.attn_bwd_workspace_size(B, H, N, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    call = sa.attn_bwd_deterministic if deterministic else sa.attn_bwd
    call(q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, B, H, N, D, scale)
    assert sa.attn_get_device_status() == 0
    assert all(_intact(b[0]) for b in bufs), "a store escaped a gradient tensor"
    to = lambda t: t.float().cpu().numpy()
    return {"dq": to(dq), "dk": to(dk), "dv": to(dv), "o": to(o)}


EDGE_N = [1, 2, 63, 64, 65, 127, 128, 129, 196, 255, 256, 257, 1000]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", EDGE_N)
def test_bwd_edge_sizes(n, d):
    inp = make_qkv(1, 3, n, d, seed=9000 + n + d)
    scale = 1.0 / math.sqrt(d)
    got = run_fwd_bwd(inp, scale)
    ref = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], scale)
    for name in ("dq", "dk", "dv"):
        if n == 1 and name in ("dq", "dk"):
            # Zero in exact arithmetic: with one key P = 1 and O = V, so dS = P (dP - D) with
            # dP = dO . V and D = dO . O the same dot product.  The kernels form the two as fp32
            # sums of d products in different orders, each within gamma_d sum_c |dO_c V_c| of
            # the exact value (gamma_d = d u / (1 - d u), u = 2^-24); dQ = scale dS K and
            # dK = scale dS^T Q carry that, then one bf16 rounding.
            u = 2.0 ** -24
            gamma = d * u / (1 - d * u)
            dov = (inp["do"].double().abs() * inp["v"].double().abs()).sum(-1, keepdim=True).numpy()
            other = (inp["k"] if name == "dq" else inp["q"]).double().abs().numpy()
            bound = scale * 2.02 * gamma * dov * other * (1 + 2.0 ** -8)
            assert (np.abs(got[name]) <= bound).all(), f"N=1 d={d} {name}: {np.abs(got[name]).max():.3g}"
            continue
        check_grad(name, got[name], ref[name], f"N={n} d={d}")


@pytest.mark.parametrize("b,h,n", [(1, 96, 200), (1, 80, 256), (2, 40, 97)])
def test_bwd_whole_heads(b, h, n):
    """d_k = 64, N <= 256 over one head per CTA at most: the single whole-head kernel (dQ
    accumulated on chip, no atomics) runs for attn_bwd and attn_bwd_deterministic alike, so
    the two give the same bits, run after run; sampled heads against the oracle."""
    inp = make_qkv(b, h, n, 64, seed=9700 + n)
    scale = 0.125
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = sa.forward(q, k, v, scale)
    outs = []
    for det in (False, True, False):
        outs.append(sa.backward(q, k, v, o, do, lse, scale, deterministic=det))
        assert sa.attn_get_device_status() == 0
    for a, c in zip(outs[0], outs[1]):
        assert torch.equal(a, c)
    for a, c in zip(outs[0], outs[2]):
        assert torch.equal(a, c)
    dq, dk, dv = (t.float().cpu().numpy() for t in outs[0])
    bh = b * h
    for idx in (0, bh // 2, bh - 1):
        bi, hi = divmod(idx, h)
        one = {x: inp[x][bi:bi + 1, hi:hi + 1] for x in ("q", "k", "v", "do")}
        ref = oracle.bwd(one["q"], one["k"], one["v"], one["do"], scale)
        got = {"dq": dq[bi:bi + 1, hi:hi + 1], "dk": dk[bi:bi + 1, hi:hi + 1], "dv": dv[bi:bi + 1, hi:hi + 1]}
        for name in ("dq", "dk", "dv"):
            check_grad(name, got[name], ref[name], f"whole heads {b}x{h}x{n} head {idx}")


@pytest.mark.parametrize("n", [4097, 4200])
def test_bwd_d64_long_sequence(n):
    """d_k = 64 past 4096 keys runs the one-CTA-per-key-block kernel instead of the persistent
    one that the shorter sizes above use; ragged last tiles in both directions."""
    inp = make_qkv(1, 2, n, 64, seed=9500 + n)
    scale = 0.125
    got = run_fwd_bwd(inp, scale)
    ref = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], scale)
    for name in ("dq", "dk", "dv"):
        check_grad(name, got[name], ref[name], f"N={n} d=64")


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_wide_logits_and_scale(d):
    inp = make_qkv(2, 2, 700, d, seed=21, qk_std=2.0)
    for scale in (1.0 / math.sqrt(d), 0.37):
        got = run_fwd_bwd(inp, scale)
        ref = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], scale)
        for name in ("dq", "dk", "dv"):
            check_grad(name, got[name], ref[name], f"d={d} scale={scale}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("deterministic", [False, True])
def test_bwd_identities_on_gpu(d, deterministic):
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i hold for the GPU gradients too.  And moving
    every key by one vector w adds scale q_i . w to a whole row of logits, which moves no weight:
    dV = P^T dO and dK = scale dS^T Q stay, and so does dQ = scale dS K, since every row of dS
    sums to 0 (up to the bf16 rounding of the shifted keys)."""
    inp = make_qkv(2, 3, 517, d, seed=22)
    scale = 1.0 / math.sqrt(d)
    got = run_fwd_bwd(inp, scale, deterministic)
    dk_sum = got["dk"].sum(axis=2)
    assert np.abs(dk_sum).max() <= 2e-2 * np.abs(got["dk"]).max() * math.sqrt(517)
    dv_sum = got["dv"].sum(axis=2)
    do_sum = inp["do"].double().sum(dim=2).numpy()
    assert np.abs(dv_sum - do_sum).max() <= 1e-2 * max(np.abs(do_sum).max(), 1.0)
    w = torch.linspace(-1.0, 1.0, d)
    shifted = dict(inp, k=(inp["k"].float() + w).bfloat16())
    got2 = run_fwd_bwd(shifted, scale, deterministic)
    for name in ("dq", "dk", "dv"):
        check_grad(f"{name} (key shift)", got2[name], got[name].astype(np.float64), f"d={d}")


def test_bwd_dk_dv_deterministic():
    inp = make_qkv(1, 4, 777, 64, seed=23)
    a = run_fwd_bwd(inp, 0.125)
    b = run_fwd_bwd(inp, 0.125)
    np.testing.assert_array_equal(a["dk"], b["dk"])
    np.testing.assert_array_equal(a["dv"], b["dv"])
    check_grad("dq", a["dq"], b["dq"].astype(np.float64), "repeat")


def test_bwd_workspace_errors():
    inp = make_qkv(1, 2, 100, 64, seed=24)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = sa.forward(q, k, v)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    need = sa.attn_bwd_workspace_size(1, 2, 100, 64)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(sa.AttnError) as e:
        sa.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, need - 16, 1, 2, 100, 64, 0.125)
    assert e.value.code == 6
    with pytest.raises(sa.AttnError) as e:
        sa.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws[16:], need - 16, 1, 2, 100, 64, 0.125)
    assert e.value.code == 6
    with pytest.raises(sa.AttnError) as e:   # an output aliasing an input
        sa.attn_bwd(q, k, v, o, do, lse, q, dk, dv, ws, need, 1, 2, 100, 64, 0.125)
    assert e.value.code == 1


def test_autograd_function():
    inp = make_qkv(1, 2, 150, 64, seed=25)
    q, k, v = (inp[x].cuda().requires_grad_(True) for x in ("q", "k", "v"))
    o = sa.attention(q, k, v)
    o.backward(inp["do"].cuda())
    ref = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], 0.125)
    for name, t in (("dq", q), ("dk", k), ("dv", v)):
        check_grad(name, t.grad.float().cpu().numpy(), ref[name], "autograd")


@pytest.mark.parametrize("shape", [(4, 8, 196, 64), (2, 8, 576, 64), (2, 4, 300, 128)])
def test_bwd_repeatable_partial_tiles(shape):
    """dQ is accumulated with fp32 atomics, so its low bits may differ between runs; but every
    head must meet the bound on its own, and repeated runs must agree far more closely than
    the bound.  The shapes end in a partial query tile, where a reuse race in the dQ staging
    buffers would corrupt whole 32-row blocks of some heads in some runs only."""
    B, H, N, D = shape
    inp = make_qkv(B, H, N, D, seed=8100 + N + D, with_do=True)
    scale = 1.0 / math.sqrt(D)
    ref = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], scale)
    runs = [run_fwd_bwd(inp, scale) for _ in range(4)]
    for r in runs:
        for name in ("dq", "dk", "dv"):
            for b in range(B):
                for h in range(H):
                    rf = rel_fro(r[name][b, h].astype(np.float64), ref[name][b, h])
                    assert rf <= GRAD_REL_FRO, f"{shape} {name} head ({b},{h}): {rf:.3g}"
        assert rel_fro(r["dq"].astype(np.float64), runs[0]["dq"].astype(np.float64)) <= 1e-3
        np.testing.assert_array_equal(r["dk"], runs[0]["dk"])
        np.testing.assert_array_equal(r["dv"], runs[0]["dv"])


@pytest.mark.parametrize("name", ["vit_b16_batch", "vit_b_mhsa_block"])
def test_bwd_workload_full(name):
    w = WORKLOADS[name]
    inp = make_workload_inputs(w)
    got = run_fwd_bwd(inp, w.scale)
    if name == "vit_b_mhsa_block":   # a spread of 24 of the 384 heads, every element
        sel = np.linspace(0, w.bh - 1, 24).astype(int)
        pick = lambda t: t.reshape(w.bh, w.N, w.d)[sel][None]
        ref = oracle.bwd(*(pick(inp[x]) for x in ("q", "k", "v", "do")), w.scale)
        got = {n_: pick(torch.from_numpy(got[n_])).numpy() for n_ in ("dq", "dk", "dv")}
    else:
        ref = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], w.scale)
    for n_ in ("dq", "dk", "dv"):
        check_grad(n_, got[n_], ref[n_], name)


@pytest.mark.parametrize("name", ["vit_l_highres", "long_text"])
def test_bwd_workload_sampled(name):
    """Full-size workloads in the benchmark's launch configuration; sampled query and key rows
    of some heads against the oracle's row-wise backward."""
    w = WORKLOADS[name]
    inp = make_workload_inputs(w)
    got = run_fwd_bwd(inp, w.scale)
    heads = [(0, 0), (w.B - 1, w.H - 1)] if name == "vit_l_highres" else [(w.B - 1, w.H // 2)]
    rng = np.random.default_rng(2)
    for (b, h) in heads:
        qrows = np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, 40)]))
        krows = np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, 40)]))
        dq, dk, dv = oracle.bwd_rows(inp["q"][b, h], inp["k"][b, h], inp["v"][b, h],
                                     inp["do"][b, h], qrows, krows, w.scale)
        where = f"{name} head ({b},{h})"
        check_grad("dq", got["dq"][b, h, qrows], dq, where)
        check_grad("dk", got["dk"][b, h, krows], dk, where)
        check_grad("dv", got["dv"][b, h, krows], dv, where)


def test_wait_timeout_reports_status():
    """A kernel wait that nobody satisfies gives up after its limit and the next status read
    reports ATTN_ERR_TIMEOUT; the context stays usable."""
    assert sa.attn_get_device_status() == 0
    sa.attn_debug_wait_timeout(2000)
    assert sa.attn_get_device_status() == 5
    assert sa.attn_get_device_status() == 0
    inp = make_qkv(1, 1, 64, 64, seed=26, with_do=False)
    o, lse = sa.forward(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda())
    torch.cuda.synchronize()
    assert sa.attn_get_device_status() == 0


def test_bwd_phases_match_single_call():
    """attn_bwd_preprocess + attn_bwd_main + attn_bwd_dq_convert == attn_bwd."""
    inp = make_qkv(2, 2, 321, 128, seed=27)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    B, H, N, D = q.shape
    o, lse = sa.forward(q, k, v)
    dq1, dk1, dv1 = sa.backward(q, k, v, o, do, lse)
    nbytes = sa.attn_bwd_workspace_size(B, H, N, D)
    ws = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")   # garbage on entry
    dq2, dk2, dv2 = (torch.empty_like(q) for _ in range(3))
    sa.attn_bwd_preprocess(o, do, lse, ws, nbytes, B, H, N, D)
    sa.attn_bwd_main(q, k, v, do, dk2, dv2, ws, nbytes, B, H, N, D, 1 / math.sqrt(D))
    sa.attn_bwd_dq_convert(ws, nbytes, dq2, B, H, N, D, 1 / math.sqrt(D))
    assert sa.attn_get_device_status() == 0
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    check_grad("dq", dq2.float().cpu().numpy(), dq1.double().cpu().numpy(), "phases")


# ------------------------------------------------------------------ deterministic dQ pass
def run_det(inp, scale):
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    B, H, N, D = q.shape
    o, lse = sa.forward(q, k, v, scale)
    bufs = [_guarded((B, H, N, D), torch.bfloat16) for _ in range(3)]
    dq, dk, dv = (b[1] for b in bufs)
    ws_bytes = sa.attn_bwd_workspace_size(B, H, N, D)
    ws = torch.full((ws_bytes,), 0x7F, dtype=torch.uint8, device="cuda")
    sa.attn_bwd_deterministic(q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, B, H, N, D, scale)
    assert sa.attn_get_device_status() == 0
    assert all(_intact(b[0]) for b in bufs), "a store escaped a gradient tensor"
    to = lambda t: t.float().cpu().numpy()
    return {"dq": to(dq), "dk": to(dk), "dv": to(dv)}


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 2, 63, 64, 65, 129, 196, 257, 1000])
def test_det_edge_sizes(n, d):
    inp = make_qkv(1, 3, n, d, seed=9500 + n + d)
    scale = 1.0 / math.sqrt(d)
    got = run_det(inp, scale)
    ref = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], scale)
    for name in ("dq", "dk", "dv"):
        if n == 1 and name in ("dq", "dk"):
            assert np.abs(got[name]).max() <= 1e-6
            continue
        check_grad(name, got[name], ref[name], f"deterministic N={n} d={d}")


def test_det_bitwise_repeatable_and_close_to_atomic():
    inp = make_qkv(2, 3, 900, 128, seed=41, qk_std=2.0)
    a, b = run_det(inp, 0.0884), run_det(inp, 0.0884)
    for name in ("dq", "dk", "dv"):
        np.testing.assert_array_equal(a[name], b[name])
    atomic = run_fwd_bwd(inp, 0.0884)
    np.testing.assert_array_equal(a["dk"], atomic["dk"])
    np.testing.assert_array_equal(a["dv"], atomic["dv"])
    check_grad("dq", a["dq"], atomic["dq"].astype(np.float64), "deterministic vs atomic")


@pytest.mark.parametrize("name", ["vit_b16_batch", "long_text"])
def test_det_workloads(name):
    w = WORKLOADS[name]
    inp = make_workload_inputs(w)
    got = run_det(inp, w.scale)
    if name == "vit_b16_batch":
        ref = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["do"], w.scale)
        for n_ in ("dq", "dk", "dv"):
            check_grad(n_, got[n_], ref[n_], name)
        return
    rng = np.random.default_rng(3)
    b, h = 0, w.H - 1
    qrows = np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, 40)]))
    krows = np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, 40)]))
    dq, dk, dv = oracle.bwd_rows(inp["q"][b, h], inp["k"][b, h], inp["v"][b, h], inp["do"][b, h],
                                 qrows, krows, w.scale)
    check_grad("dq", got["dq"][b, h, qrows], dq, name)
    check_grad("dk", got["dk"][b, h, krows], dk, name)
    check_grad("dv", got["dv"][b, h, krows], dv, name)
