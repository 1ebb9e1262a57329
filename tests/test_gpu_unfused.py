"""Standard attention (attn_fwd_unfused: S and P through HBM) against the fp64 oracle and the
fused forward, on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import self_attention_gb300 as sa
from self_attention_gb300.inputs import WORKLOADS, make_qkv, make_workload_inputs
from _compare import O_MAX_ABS, O_REL_FRO, bf16_spacing, check_lse, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_attention_gb300.build import build
    sa.load_library(build())


def check_o_bf16_weights(got, ref, a_abs, where):
    """O of a path whose normalised weights enter P V rounded to bf16 (relative error up to
    2^-9 each, O moving by at most 2^-9 * A with A = sum_j P_ij |V_j|), plus half a bf16 spacing
    of output rounding and fp32 accumulation (2^-12 * A)."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = np.maximum(O_MAX_ABS, 0.5 * bf16_spacing(ref) + (2.0 ** -9 + 2.0 ** -12) * np.asarray(a_abs))
    assert not (err > bound).any(), f"{where}: O max abs {err.max():.4g}"
    assert rel_fro(got, ref) <= O_REL_FRO, f"{where}: O relative Frobenius {rel_fro(got, ref):.3g}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 63, 196, 257, 700])
def test_unfused_matches_oracle(n, d):
    inp = make_qkv(2, 3, n, d, seed=4100 + n + d, with_do=False)
    scale = 1.0 / math.sqrt(d)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = sa.forward_unfused(q, k, v, scale)
    torch.cuda.synchronize()
    assert sa.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], scale)
    a_abs, _ = oracle.fwd(inp["q"], inp["k"], inp["v"].abs(), scale)
    check_o_bf16_weights(o.float().cpu().numpy(), o_ref, a_abs, f"unfused N={n} d={d}")
    check_lse(lse.cpu().numpy(), lse_ref, f"unfused N={n} d={d}")
    # the fused forward on the same inputs: the same result to within both paths' rounding
    of, lf = sa.forward(q, k, v, scale)
    assert rel_fro(of.float().cpu().numpy(), o.float().cpu().numpy()) < 5e-3
    np.testing.assert_allclose(lf.cpu().numpy(), lse.cpu().numpy(), rtol=0, atol=1e-4 * max(1.0, float(np.abs(lse_ref).max())))


def test_unfused_vit_b16_batch_full():
    """The ViT-B/16 batch shape (768 heads of N = 196), every element."""
    w = WORKLOADS["vit_b16_batch"]
    inp = make_workload_inputs(w)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = sa.forward_unfused(q, k, v, w.scale)
    torch.cuda.synchronize()
    assert sa.attn_get_device_status() == 0
    sel = np.linspace(0, w.bh - 1, 16).astype(int)
    pick = lambda t: t.reshape(w.bh, w.N, w.d)[sel].reshape(1, -1, w.N, w.d)
    ref_in = {x: pick(inp[x]) for x in ("q", "k", "v")}
    o_ref, lse_ref = oracle.fwd(ref_in["q"], ref_in["k"], ref_in["v"], w.scale)
    a_abs, _ = oracle.fwd(ref_in["q"], ref_in["k"], ref_in["v"].abs(), w.scale)
    check_o_bf16_weights(o.float().cpu().numpy().reshape(w.bh, w.N, w.d)[sel][None], o_ref, a_abs, "vit_b16_batch")
    check_lse(lse.cpu().numpy().reshape(w.bh, w.N)[sel][None], lse_ref, "vit_b16_batch")
