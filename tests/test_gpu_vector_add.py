"""Section 2's vector add on the GPU (the library's HBM probe) against the fp32 oracle: every
element bit for bit, at sizes around the 4-element vector width and the wave size."""
import numpy as np
import pytest
import torch

import oracle
import self_attention_gb300 as sa

pytestmark = pytest.mark.gpu

GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_attention_gb300.build import build
    sa.load_library(build())


def _draw(n, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, generator=g) * 10).float(), (torch.randn(n, generator=g) * 10).float()


@pytest.mark.parametrize("n", [1, 3, 4, 5, 255, 256, 1023, 1024, 1025, 4097, 152 * 2048 + 7,
                               (1 << 22) + 3, 40_000_003])
def test_vector_add_bitwise(n):
    a, b = _draw(n, seed=n)
    buf = torch.full((n + 2 * GUARD,), float("nan"), device="cuda")
    c = buf[GUARD:GUARD + n]
    sa.vector_add(a.cuda(), b.cuda(), c, n)
    torch.cuda.synchronize()
    ref = oracle.vector_add(a.numpy(), b.numpy())
    np.testing.assert_array_equal(c.cpu().numpy(), ref)
    assert torch.isnan(buf[:GUARD]).all() and torch.isnan(buf[-GUARD:]).all()


def test_vector_add_in_place():
    n = 100_001
    a, b = _draw(n, seed=1)
    ad = a.cuda()
    sa.vector_add(ad, b.cuda(), ad, n)
    np.testing.assert_array_equal(ad.cpu().numpy(), oracle.vector_add(a.numpy(), b.numpy()))
