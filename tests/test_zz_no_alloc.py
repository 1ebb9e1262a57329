"""attn_bwd_noalloc: the backward pass for callers that cannot allocate device memory when
they run it (a fixed memory budget, or a framework that owns every device allocation).  Its
scratch is a fixed 64 MiB array inside the library instead of a caller-supplied workspace.

This file is collected last on purpose, so that a run stopping at its first failure has run
every other test before this one.  It passes on its own in a fresh process and after the others.
"""
import math

import pytest
import torch

import self_attention_gb300 as sa
from self_attention_gb300.inputs import make_qkv
from _compare import check_grad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_attention_gb300.build import build
    sa.load_library(build())


def test_noalloc_matches_attn_bwd_on_two_calls_in_a_row():
    """Two consecutive calls (different sizes, so the second sees the first one's leftovers in
    the shared scratch) agree with attn_bwd: dK and dV bit for bit, dQ (accumulated with fp32
    atomics in either path) within the gradient tolerance used by every other test."""
    for B, H, N, D, seed in ((2, 3, 517, 128, 31), (1, 4, 300, 64, 32)):
        inp = make_qkv(B, H, N, D, seed=seed)
        q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
        scale = 1.0 / math.sqrt(D)
        o, lse = sa.forward(q, k, v, scale)
        dq1, dk1, dv1 = sa.backward(q, k, v, o, do, lse, scale)
        dq2, dk2, dv2 = (torch.empty_like(q) for _ in range(3))
        sa.attn_bwd_noalloc(q, k, v, o, do, lse, dq2, dk2, dv2, B, H, N, D, scale)
        assert sa.attn_get_device_status() == 0
        assert torch.equal(dk1, dk2), f"dK differs (N={N}, d={D})"
        assert torch.equal(dv1, dv2), f"dV differs (N={N}, d={D})"
        check_grad("dq", dq2.float().cpu().numpy(), dq1.double().cpu().numpy(),
                   f"noalloc N={N} d={D}")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    """B=2, H=16, N=16384, d=128 needs ~272 MB of scratch: refused before anything runs."""
    assert sa.attn_bwd_workspace_size(2, 16, 16384, 128) > 64 << 20
    with pytest.raises(sa.AttnError) as e:
        sa.attn_bwd_noalloc(0, 0, 0, 0, 0, 0, 0, 0, 0, 2, 16, 16384, 128, 0.088)
    assert e.value.code == 8
    assert "ATTN_ERR_TOO_LARGE" in str(e.value)
