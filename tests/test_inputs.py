"""The seeded input recipe, on CPU: the one module the oracle and the GPU path share.  Same
seed, same bits; draws in the order Q, K, V, dO; N(0, std^2) values rounded to bf16; the five
workloads' shapes and distributions; the block workload's head split of X W."""
import dataclasses
import math

import pytest
import torch

from self_attention_gb300.inputs import WORKLOADS, make_block_inputs, make_qkv, make_workload_inputs


def test_same_seed_same_bits_and_other_seeds_differ():
    a = make_qkv(2, 3, 70, 64, seed=7)
    b = make_qkv(2, 3, 70, 64, seed=7)
    c = make_qkv(2, 3, 70, 64, seed=8)
    for x in ("q", "k", "v", "do"):
        assert a[x].dtype == torch.bfloat16 and a[x].shape == (2, 3, 70, 64) and a[x].is_contiguous()
        assert torch.equal(a[x].view(torch.int16), b[x].view(torch.int16))
        assert not torch.equal(a[x], c[x])


def test_draw_order_is_q_k_v_do_from_one_generator():
    d = make_qkv(1, 2, 33, 64, seed=11, qk_std=2.0, v_std=1.0)
    gen = torch.Generator(device="cpu").manual_seed(11)
    shape = (1, 2, 33, 64)
    for x, std in (("q", 2.0), ("k", 2.0), ("v", 1.0), ("do", 1.0)):
        ref = torch.randn(shape, generator=gen, dtype=torch.float32) * std
        assert torch.equal(d[x], ref.to(torch.bfloat16)), x


@pytest.mark.parametrize("std", [1.0, 2.0])
def test_values_are_gaussian_with_the_stated_deviation(std):
    d = make_qkv(4, 4, 256, 64, seed=3, qk_std=std, with_do=False)
    q = d["q"].double()
    n = q.numel()
    assert abs(q.mean().item()) < 5 * std / math.sqrt(n)
    assert q.std().item() == pytest.approx(std, rel=0.01)
    # about 68.3 % within one deviation (bf16 rounding moves a few values across the edge)
    assert (q.abs() <= std).double().mean().item() == pytest.approx(0.6827, abs=0.01)


def test_workload_table():
    got = {n: (w.B, w.H, w.N, w.d, w.qk_std, w.v_std, w.backward, w.model_dim) for n, w in WORKLOADS.items()}
    assert got == {
        "vit_b16_single": (1, 12, 196, 64, 1.0, 1.0, False, 0),
        "vit_b16_batch": (64, 12, 196, 64, 1.0, 1.0, True, 0),
        "vit_l_highres": (8, 16, 4096, 64, 1.0, 1.0, True, 0),
        "long_text": (2, 16, 16384, 128, 2.0, 1.0, True, 0),
        "vit_b_mhsa_block": (32, 12, 576, 64, 1.0, 1.0, True, 768),
    }
    assert len({w.seed for w in WORKLOADS.values()}) == len(WORKLOADS)
    for w in WORKLOADS.values():
        assert w.scale == float(torch.tensor(1 / math.sqrt(w.d), dtype=torch.float32))
        assert w.fwd_flops() == 4.0 * w.B * w.H * w.N ** 2 * w.d
        assert w.bwd_flops() == 10.0 * w.B * w.H * w.N ** 2 * w.d


def test_block_inputs_split_the_projection_into_heads():
    w = WORKLOADS["vit_b_mhsa_block"]
    w = dataclasses.replace(w, B=2, N=9)    # the recipe at a small size
    d = make_block_inputs(w)
    assert d["x"].shape == (2, 9, 768) and d["w_q"].shape == (768, 768)
    assert d["w_q"].double().std().item() == pytest.approx(1 / math.sqrt(768), rel=0.02)
    for name, wm in (("q", "w_q"), ("k", "w_k"), ("v", "w_v")):
        full = (d["x"].float() @ d[wm].float())                 # [B, N, 768]
        for h in (0, 5, 11):
            ref = full[:, :, 64 * h:64 * (h + 1)].to(torch.bfloat16)
            assert torch.equal(d[name][:, h], ref), (name, h)
    assert d["do"].shape == (2, 12, 9, 64)
    assert torch.equal(make_workload_inputs(w)["q"], d["q"])
