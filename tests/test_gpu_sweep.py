"""Seeded sweep over random shapes: forward and both backward modes against the oracle on a
few heads of each.  The sizes span the kernel variants the dispatch picks (one CTA per tile or
persistent CTAs walking several items, short and long sequences, ragged last tiles of queries
and keys) and two logit spreads."""
import math

import numpy as np
import pytest
import torch

import oracle
import self_attention_gb300 as sa
from self_attention_gb300.inputs import make_qkv
from _compare import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


def _shapes():
    """d_k in {64, 128} x {few, some, many heads (more tiles than resident CTAs)} x two random
    sequence lengths, logit spreads alternating."""
    rng = np.random.default_rng(20261203)
    out = []
    for d in (64, 128):
        for heads in (3, 40, 320):
            for _ in range(2):
                n = int(rng.integers(1, 1200))
                H = int(rng.choice([1, 2, 4, 8]))
                B = max(1, heads // H)
                out.append((B, H, n, d, 1.0 + (len(out) % 2)))
        # long sequences (at d_k = 64 past 4096 the one-CTA-per-key-block backward)
        out.append((1, 2, int(rng.integers(4100, 5200)), d, 2.0))
    return out


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_attention_gb300.build import build
    sa.load_library(build())


@pytest.mark.parametrize("shape", _shapes(), ids=lambda s: "B%dH%dN%dd%ds%g" % s)
def test_sweep(shape):
    B, H, N, D, std = shape
    scale = 1.0 / math.sqrt(D)
    inp = make_qkv(B, H, N, D, seed=31000 + N + D + B * H, qk_std=std)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = sa.forward(q, k, v, scale)
    grads = sa.backward(q, k, v, o, do, lse, scale)
    grads_det = sa.backward(q, k, v, o, do, lse, scale, deterministic=True)
    torch.cuda.synchronize()
    assert sa.attn_get_device_status() == 0
    # first and last head in full (with several heads, the last one sits in another CTA's item)
    for (b, h) in {(0, 0), (B - 1, H - 1)}:
        one = {x: inp[x][b:b + 1, h:h + 1] for x in ("q", "k", "v", "do")}
        o_ref, lse_ref = oracle.fwd(one["q"], one["k"], one["v"], scale)
        a_abs, _ = oracle.fwd(one["q"], one["k"], one["v"].abs(), scale)
        where = f"{shape} head ({b},{h})"
        check_o(o[b:b + 1, h:h + 1].float().cpu().numpy(), o_ref, a_abs, where)
        check_lse(lse[b:b + 1, h:h + 1].cpu().numpy(), lse_ref, where)
        ref = oracle.bwd(one["q"], one["k"], one["v"], one["do"], scale)
        for mode, gs in (("atomic", grads), ("deterministic", grads_det)):
            for name, t in zip(("dq", "dk", "dv"), gs):
                got = t[b:b + 1, h:h + 1].float().cpu().numpy()
                if N == 1 and name in ("dq", "dk"):   # exactly zero: compare absolutely
                    assert np.abs(got).max() <= 1e-6, f"{where} {mode} {name}"
                    continue
                check_grad(name, got, ref[name], f"{where} {mode}")
