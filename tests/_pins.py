"""Pins for the fp64 oracle: checks against facts fixed by the article's formulas and by
mathematics, never against the oracle itself.

Each pin takes an oracle library handle (``oracle.load_library(path)``) so that the same
pins can be run against deliberately broken copies of the oracle (tests/test_oracle_mutants.py)
and shown to catch them.  A pin raises AssertionError when the fact does not hold.

Formulas ("Self-attention, CUDA kernels and FlashAttention", section 1):
S = Q K^T / sqrt(d_k); P = row softmax of S (each row sums to one); O = P V; heads independent.
Section 3 ("Recomputation in backpropagation"): the saved statistic is per row; here the
natural-log log-sum-exp of the row of S.  Backward: chain rule on the same formulas.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def pin_rows_sum_to_one(lib):
    """With d_k = N and V = identity, O is P itself: every row is non-negative and sums to 1
    (section 1, softmax weighting)."""
    rng = _rng(1)
    n = 24
    q, k = _rand(rng, 1, 2, n, n), _rand(rng, 1, 2, n, n)
    v = np.broadcast_to(np.eye(n), (1, 2, n, n)).copy()
    o, _ = oracle.fwd(q, k, v, 1.0 / math.sqrt(n), lib=lib)
    assert (o >= 0).all()
    np.testing.assert_allclose(o.sum(-1), 1.0, rtol=0, atol=1e-12)


def pin_probabilities_match_library_softmax(lib):
    """P (read through V = identity) equals torch.softmax of the scaled scores, fp64."""
    import torch
    rng = _rng(2)
    n = 17
    q, k = _rand(rng, 1, 1, n, n), _rand(rng, 1, 1, n, n)
    v = np.eye(n)[None, None]
    scale = 0.3
    o, lse = oracle.fwd(q, k, v, scale, lib=lib)
    qt, kt = torch.from_numpy(q), torch.from_numpy(k)
    s = (qt @ kt.transpose(-1, -2)) * scale
    np.testing.assert_allclose(o, torch.softmax(s, -1).numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def pin_zero_queries_average_values(lib):
    """Q = 0 makes every score 0: each output row is the mean of V's rows and LSE = log N."""
    rng = _rng(3)
    for n, d in ((1, 4), (7, 8), (65, 16)):
        q = np.zeros((2, 3, n, d))
        k, v = _rand(rng, 2, 3, n, d), _rand(rng, 2, 3, n, d)
        o, lse = oracle.fwd(q, k, v, 1.0 / math.sqrt(d), lib=lib)
        np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, math.log(n), rtol=0, atol=1e-13)


def pin_dominant_key_selects_its_value(lib):
    """A key whose score beats every other by > 400 takes all the weight: O_i = V_{j*} and
    LSE_i = S_{i j*} to rounding."""
    rng = _rng(4)
    n, d, jstar = 33, 4, 21
    q = _rand(rng, 1, 1, n, d, std=0.1)
    q[..., 0] = 1.0 + np.abs(q[..., 0])           # every query has a large first component
    k = _rand(rng, 1, 1, n, d, std=0.01)
    k[0, 0, jstar] = [2000.0, 0.0, 0.0, 0.0]
    v = _rand(rng, 1, 1, n, d)
    scale = 0.5
    o, lse = oracle.fwd(q, k, v, scale, lib=lib)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0, jstar], (n, d)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], scale * q[0, 0] @ k[0, 0, jstar], rtol=1e-15, atol=1e-12)


def pin_joint_key_value_permutation(lib):
    """Permuting the rows of K and V together leaves O and LSE unchanged (the sum over j does
    not depend on the order of the keys)."""
    rng = _rng(5)
    n, d = 40, 8
    q, k, v = (_rand(rng, 2, 2, n, d) for _ in range(3))
    perm = rng.permutation(n)
    o1, l1 = oracle.fwd(q, k, v, 0.35, lib=lib)
    o2, l2 = oracle.fwd(q, k[:, :, perm], v[:, :, perm], 0.35, lib=lib)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)
    # permuting queries permutes the output rows
    o3, l3 = oracle.fwd(q[:, :, perm], k, v, 0.35, lib=lib)
    np.testing.assert_allclose(o3, o1[:, :, perm], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l3, l1[:, :, perm], rtol=0, atol=1e-12)


def pin_key_shift(lib):
    """K -> K + 1 w^T adds scale * q_i . w to every score of row i: softmax ignores a per-row
    constant, so O is unchanged and LSE_i grows by exactly that constant."""
    rng = _rng(6)
    n, d, scale = 19, 8, 0.25
    q, k, v = (_rand(rng, 1, 2, n, d) for _ in range(3))
    w = _rand(rng, d)
    o1, l1 = oracle.fwd(q, k, v, scale, lib=lib)
    o2, l2 = oracle.fwd(q, k + w, v, scale, lib=lib)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + scale * (q @ w), rtol=0, atol=1e-12)


def pin_value_affine(lib):
    """V -> a V + 1 b^T maps O -> a O + 1 b^T because each row of P sums to one."""
    rng = _rng(7)
    n, d = 23, 8
    q, k, v = (_rand(rng, 1, 1, n, d) for _ in range(3))
    a, b = -1.7, _rand(rng, d)
    o1, _ = oracle.fwd(q, k, v, 0.4, lib=lib)
    o2, _ = oracle.fwd(q, k, a * v + b, 0.4, lib=lib)
    np.testing.assert_allclose(o2, a * o1 + b, rtol=0, atol=1e-12)


def pin_single_token(lib):
    """N = 1: the one weight is 1, so O = V, LSE = scale q.k, dQ = dK = 0 and dV = dO."""
    rng = _rng(8)
    d, scale = 8, 0.125
    q, k, v, do = (_rand(rng, 2, 3, 1, d) for _ in range(4))
    o, lse = oracle.fwd(q, k, v, scale, lib=lib)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, scale * (q * k).sum(-1), rtol=0, atol=1e-14)
    g = oracle.bwd(q, k, v, do, scale, lib=lib)
    np.testing.assert_allclose(g["dq"], 0.0, atol=1e-14)
    np.testing.assert_allclose(g["dk"], 0.0, atol=1e-14)
    np.testing.assert_allclose(g["dv"], do, rtol=0, atol=1e-14)


def pin_two_tokens_sigmoid(lib):
    """N = 2: the weight on key 0 is the logistic function of the score difference."""
    rng = _rng(9)
    d, scale = 4, 0.6
    q, k, v = (_rand(rng, 1, 1, 2, d) for _ in range(3))
    o, lse = oracle.fwd(q, k, v, scale, lib=lib)
    for i in range(2):
        s0 = scale * q[0, 0, i] @ k[0, 0, 0]
        s1 = scale * q[0, 0, i] @ k[0, 0, 1]
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        np.testing.assert_allclose(o[0, 0, i], w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 1], atol=1e-14)
        np.testing.assert_allclose(lse[0, 0, i], max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))),
                                   atol=1e-14)


def pin_heads_independent(lib):
    """Each head is computed on its own (section 1, multi-head): reordering heads reorders the
    results, and a head's result does not depend on the others."""
    rng = _rng(10)
    n, d = 12, 4
    q, k, v = (_rand(rng, 2, 3, n, d) for _ in range(3))
    o, lse = oracle.fwd(q, k, v, 0.5, lib=lib)
    o1, l1 = oracle.fwd(q[1:2, 2:3], k[1:2, 2:3], v[1:2, 2:3], 0.5, lib=lib)
    np.testing.assert_array_equal(o1[0, 0], o[1, 2])
    np.testing.assert_array_equal(l1[0, 0], lse[1, 2])
    p = [2, 0, 1]
    o2, _ = oracle.fwd(q[:, p], k[:, p], v[:, p], 0.5, lib=lib)
    np.testing.assert_array_equal(o2, o[:, p])


def pin_worked_example(lib):
    """The hand-derived N=2 example in tests/golden/worked_n2_d1.json (forward and backward)."""
    with open(os.path.join(GOLDEN, "worked_n2_d1.json")) as f:
        g = json.load(f)
    arr = lambda name: np.array(g["inputs"][name], dtype=np.float64)[None, None]
    q, k, v, do = arr("q"), arr("k"), arr("v"), arr("do")
    scale = g["inputs"]["scale"]
    o, lse = oracle.fwd(q, k, v, scale, lib=lib)
    e = g["expected"]
    np.testing.assert_allclose(o[0, 0], e["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], e["lse"], rtol=0, atol=1e-14)
    r = oracle.bwd(q, k, v, do, scale, lib=lib)
    for name in ("dq", "dk", "dv"):
        np.testing.assert_allclose(r[name][0, 0], e[name], rtol=0, atol=1e-14, err_msg=name)
    np.testing.assert_allclose(r["D"][0, 0], e["D"], rtol=0, atol=1e-14)


def _loss(lib, q, k, v, do, scale):
    o, _ = oracle.fwd(q, k, v, scale, lib=lib)
    return float((o * do).sum())


def pin_finite_differences(lib):
    """Central differences of L = <dO, O> (h = 1e-6) match every entry of dQ, dK, dV."""
    rng = _rng(11)
    for n, d in ((1, 3), (3, 2), (6, 4)):
        q, k, v, do = (_rand(rng, 1, 2, n, d) for _ in range(4))
        scale = 1.0 / math.sqrt(d)
        g = oracle.bwd(q, k, v, do, scale, lib=lib)
        h = 1e-6
        for name, x in (("dq", q), ("dk", k), ("dv", v)):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = _loss(lib, q, k, v, do, scale)
                x[idx] = old - h
                lm = _loss(lib, q, k, v, do, scale)
                x[idx] = old
                fd[idx] = (lp - lm) / (2 * h)
            err = np.abs(fd - g[name]).max() / max(np.abs(fd).max(), 1e-3)
            assert err < 1e-6, f"{name}: finite-difference mismatch {err:.3g} (n={n}, d={d})"


def pin_backward_identities(lib):
    """Sum_j dK_j = 0 (adding a vector to every key changes nothing), Sum_j dV_j = Sum_i dO_i
    (adding a vector to every value adds it to every output), and D = D' (two definitions
    of rowsum(P o dP))."""
    rng = _rng(12)
    n, d = 37, 8
    q, k, v, do = (_rand(rng, 2, 2, n, d) for _ in range(4))
    g = oracle.bwd(q, k, v, do, 0.3, lib=lib)
    np.testing.assert_allclose(g["dk"].sum(2), 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dv"].sum(2), do.sum(2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["D"], g["Dprime"], rtol=0, atol=1e-12)
    # Q -> c Q with scale -> scale / c is the same function, so dQ scales by 1/c
    g2 = oracle.bwd(2.0 * q, k, v, do, 0.15, lib=lib)
    np.testing.assert_allclose(g2["dq"], g["dq"] / 2.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g2["dk"], g["dk"], rtol=0, atol=1e-12)


def pin_library_autograd(lib):
    """On tiny fp64 inputs, torch's scaled_dot_product_attention (CPU, autograd) gives the
    same O, dQ, dK and dV."""
    import torch
    rng = _rng(13)
    for n, d in ((5, 4), (13, 8)):
        q, k, v, do = (_rand(rng, 2, 2, n, d) for _ in range(4))
        scale = 1.0 / math.sqrt(d)
        ts = [torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v)]
        ot = torch.nn.functional.scaled_dot_product_attention(*ts, scale=scale)
        ot.backward(torch.from_numpy(do))
        g = oracle.bwd(q, k, v, do, scale, lib=lib)
        np.testing.assert_allclose(g["o"], ot.detach().numpy(), rtol=0, atol=1e-12)
        for name, t in zip(("dq", "dk", "dv"), ts):
            np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=0, atol=1e-12, err_msg=name)


def pin_rows_variants(lib):
    """The sampled-row entry points (used at full workload sizes) agree with the full ones
    at the sampled indices; the full ones are pinned above."""
    rng = _rng(14)
    n, d, scale = 50, 8, 0.3
    q, k, v, do = (_rand(rng, 1, 1, n, d) for _ in range(4))
    o, lse = oracle.fwd(q, k, v, scale, lib=lib)
    g = oracle.bwd(q, k, v, do, scale, lib=lib)
    rows = np.array([0, 7, 49, 23])
    o_r, l_r = oracle.fwd_rows(q[0, 0], k[0, 0], v[0, 0], rows, scale, lib=lib)
    np.testing.assert_allclose(o_r, o[0, 0, rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l_r, lse[0, 0, rows], rtol=0, atol=1e-13)
    krows = np.array([3, 49, 0])
    dq, dk, dv = oracle.bwd_rows(q[0, 0], k[0, 0], v[0, 0], do[0, 0], rows, krows, scale, lib=lib)
    np.testing.assert_allclose(dq, g["dq"][0, 0, rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, g["dk"][0, 0, krows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, g["dv"][0, 0, krows], rtol=0, atol=1e-12)


def pin_vector_add(lib):
    """Section 2's C = A + B in fp32: adding zero changes nothing, the sum is symmetric, small
    integers add exactly, x + (-x) = 0, and a tie rounds to the even neighbour
    (1 + 3 * 2^-24 lies halfway between 1 + 2^-23 and 1 + 2^-22 and must give 1 + 2^-22)."""
    rng = _rng(15)
    a = (rng.standard_normal(1001) * 3).astype(np.float32)
    b = (rng.standard_normal(1001) * 3).astype(np.float32)
    zero = np.zeros_like(a)
    np.testing.assert_array_equal(oracle.vector_add(a, zero, lib=lib), a)
    np.testing.assert_array_equal(oracle.vector_add(a, b, lib=lib), oracle.vector_add(b, a, lib=lib))
    i = np.arange(-500, 501, dtype=np.float32)
    np.testing.assert_array_equal(oracle.vector_add(i, 2 * i, lib=lib), 3 * i)
    np.testing.assert_array_equal(oracle.vector_add(a, -a, lib=lib), zero)
    one = np.ones(4, np.float32)
    tie = np.full(4, 3.0 * 2.0 ** -24, np.float32)
    np.testing.assert_array_equal(oracle.vector_add(one, tie, lib=lib),
                                  np.full(4, 1.0 + 2.0 ** -22, np.float32))
    big = np.full(3, 2.0 ** 24, np.float32)
    np.testing.assert_array_equal(oracle.vector_add(big, np.ones(3, np.float32), lib=lib), big)


def pin_qkv_projection(lib):
    """Section 1's Q = X W_Q (and K, V), head h = columns [h d_k, (h+1) d_k): W = I reproduces
    the head-split X exactly; the map is linear in W; the backward satisfies
    <dX, X> = sum_t <dW_t, W_t> (both equal sum_t <dY_t, Y_t>), matches central finite
    differences, and matches torch autograd on the same fp64 inputs."""
    import torch
    rng = _rng(16)
    B, N, D, H = 2, 5, 8, 2
    d = D // H
    x = _rand(rng, B, N, D)
    ws = [_rand(rng, D, D) for _ in range(3)]
    eye = np.eye(D)
    q, k, v = oracle.qkv_proj(x, eye, eye, eye, H)
    for h in range(H):
        np.testing.assert_array_equal(q[:, h], x[:, :, h * d:(h + 1) * d])
    w2 = _rand(rng, D, D)
    lhs = oracle.qkv_proj(x, 2.5 * ws[0] + w2, ws[1], ws[2], H)[0]
    rhs = 2.5 * oracle.qkv_proj(x, ws[0], ws[1], ws[2], H)[0] + oracle.qkv_proj(x, w2, ws[1], ws[2], H)[0]
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)
    dys = [_rand(rng, B, H, N, d) for _ in range(3)]
    dx, dwq, dwk, dwv = oracle.qkv_proj_bwd(x, *ws, *dys)
    ys = oracle.qkv_proj(x, *ws, H)
    L = sum(float((y * dy).sum()) for y, dy in zip(ys, dys))
    np.testing.assert_allclose(float((dx * x).sum()), L, rtol=1e-12)
    np.testing.assert_allclose(sum(float((dw * w).sum()) for dw, w in zip((dwq, dwk, dwv), ws)), L, rtol=1e-12)
    # finite differences on a few entries of X and W_K
    h_ = 1e-6

    def loss(xx, wk):
        yy = oracle.qkv_proj(xx, ws[0], wk, ws[2], H)
        return sum(float((y * dy).sum()) for y, dy in zip(yy, dys))
    for idx in ((0, 1, 3), (1, 4, 7)):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h_
        xm[idx] -= h_
        np.testing.assert_allclose((loss(xp, ws[1]) - loss(xm, ws[1])) / (2 * h_), dx[idx], rtol=1e-6, atol=1e-8)
    for idx in ((0, 0), (5, 2), (7, 6)):
        wp, wm = ws[1].copy(), ws[1].copy()
        wp[idx] += h_
        wm[idx] -= h_
        np.testing.assert_allclose((loss(x, wp) - loss(x, wm)) / (2 * h_), dwk[idx], rtol=1e-6, atol=1e-8)
    # torch autograd
    xt = torch.from_numpy(x.copy()).requires_grad_(True)
    wt = [torch.from_numpy(w.copy()).requires_grad_(True) for w in ws]
    out = [(xt @ w).reshape(B, N, H, d).permute(0, 2, 1, 3) for w in wt]
    sum((o * torch.from_numpy(dy)).sum() for o, dy in zip(out, dys)).backward()
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=0, atol=1e-12)
    for dw, w in zip((dwq, dwk, dwv), wt):
        np.testing.assert_allclose(dw, w.grad.numpy(), rtol=0, atol=1e-12)


ALL_PINS = [
    pin_rows_sum_to_one,
    pin_probabilities_match_library_softmax,
    pin_zero_queries_average_values,
    pin_dominant_key_selects_its_value,
    pin_joint_key_value_permutation,
    pin_key_shift,
    pin_value_affine,
    pin_single_token,
    pin_two_tokens_sigmoid,
    pin_heads_independent,
    pin_worked_example,
    pin_finite_differences,
    pin_backward_identities,
    pin_library_autograd,
    pin_rows_variants,
    pin_vector_add,
    pin_qkv_projection,
]
