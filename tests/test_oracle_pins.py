"""Pins for the CPU oracle: each test ties it to something other than itself.

- finite differences of L = sum(O * dO) (the gradient-check method of
  "A transformer in PTX", §Checking the gradients), along a random direction
  and along the gradient, for q, k and v;
- rows of P sum to one, with exact zeros above the diagonal;
- causality: keys/values after position t cannot change O_t or LSE_t;
- grouped-query attention equals multi-head attention with K/V heads
  repeated, and its dK/dV are the group sums;
- closed forms (first row, constant keys, one token);
- a three-token example worked by hand (tests/golden);
- torch's own float64 CPU attention with autograd (a library special case).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def rand(shape, rng, std=1.0):
    return np.ascontiguousarray(rng.standard_normal(shape) * std)


def rand_case(B, T, Hq, Hkv, d, seed, std=1.0):
    rng = np.random.default_rng(seed)
    return (rand((B, T, Hq, d), rng, std), rand((B, T, Hkv, d), rng, std), rand((B, T, Hkv, d), rng),
            rand((B, T, Hq, d), rng))


def loss(q, k, v, dout, causal, scale=None):
    o, _ = oracle.fwd(q, k, v, causal=causal, scale=scale)
    return float(np.sum(o * dout))


# ---------------------------------------------------------------- finite differences
FD_SHAPES = [
    (2, 9, 4, 2, 12),   # the page's awkward gradient-check sizes: 4 query heads of 12 over 2 kv heads, 9 tokens
    (1, 7, 6, 2, 5),    # three query heads per kv head
    (1, 1, 3, 1, 4),    # a single token
    (1, 13, 2, 2, 8),   # plain multi-head
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", FD_SHAPES)
def test_finite_differences(shape, causal):
    B, T, Hq, Hkv, d = shape
    q, k, v, dout = rand_case(B, T, Hq, Hkv, d, seed=7 + T + d)
    g = oracle.bwd(q, k, v, dout, causal=causal)
    rng = np.random.default_rng(99)
    eps = 1e-5
    for name, x in (("q", q), ("k", k), ("v", v)):
        grad = g["d" + name]
        directions = [rng.standard_normal(x.shape)]
        if np.linalg.norm(grad) > 0:
            directions.append(grad.copy())
        for u in directions:
            u = u / np.linalg.norm(u)
            args = {"q": q, "k": k, "v": v}
            plus = dict(args)
            minus = dict(args)
            plus[name] = x + eps * u
            minus[name] = x - eps * u
            fd = (loss(plus["q"], plus["k"], plus["v"], dout, causal)
                  - loss(minus["q"], minus["k"], minus["v"], dout, causal)) / (2 * eps)
            an = float(np.sum(grad * u))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


# ---------------------------------------------------------------- probabilities
@pytest.mark.parametrize("causal", [True, False])
def test_probability_rows(causal):
    q, k, _, _ = rand_case(2, 37, 4, 2, 16, seed=3, std=2.0)
    for b, h in ((0, 0), (1, 3)):
        P, lse = oracle.probs(q, k, b, h, causal=causal)
        assert np.allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        assert (P >= 0).all()
        if causal:
            assert np.all(np.triu(P, 1) == 0.0)
            assert np.all(np.diag(P) > 0)
        # LSE against the scores it normalises: P_ij = exp(s_ij - LSE_i)
        kv = h // 2
        s = (q[b, :, h, :] @ k[b, :, kv, :].T) / math.sqrt(16)
        i, j = 20, 5
        assert abs(P[i, j] - math.exp(s[i, j] - lse[i])) <= 1e-14


# ---------------------------------------------------------------- causality
def test_causality():
    B, T, Hq, Hkv, d = 2, 24, 4, 2, 8
    q, k, v, dout = rand_case(B, T, Hq, Hkv, d, seed=11)
    o, lse = oracle.fwd(q, k, v)
    t = 9
    rng = np.random.default_rng(5)
    k2, v2 = k.copy(), v.copy()
    k2[:, t + 1:] += rng.standard_normal(k2[:, t + 1:].shape) * 3
    v2[:, t + 1:] += rng.standard_normal(v2[:, t + 1:].shape) * 3
    o2, lse2 = oracle.fwd(q, k2, v2)
    assert np.array_equal(o[:, :t + 1], o2[:, :t + 1])
    assert np.array_equal(lse[:, :, :t + 1], lse2[:, :, :t + 1])
    assert not np.allclose(o[:, t + 1:], o2[:, t + 1:])
    # and gradients w.r.t. q at positions <= t are likewise unchanged
    g = oracle.bwd(q, k, v, dout)
    g2 = oracle.bwd(q, k2, v2, dout)
    assert np.array_equal(g["dq"][:, :t + 1], g2["dq"][:, :t + 1])


# ---------------------------------------------------------------- GQA vs repeated heads
@pytest.mark.parametrize("causal", [True, False])
def test_gqa_equals_repeated_heads(causal):
    B, T, Hq, Hkv, d = 2, 19, 6, 2, 8
    G = Hq // Hkv
    q, k, v, dout = rand_case(B, T, Hq, Hkv, d, seed=21)
    kr = np.ascontiguousarray(np.repeat(k, G, axis=2))
    vr = np.ascontiguousarray(np.repeat(v, G, axis=2))
    a = oracle.bwd(q, k, v, dout, causal=causal)
    r = oracle.bwd(q, kr, vr, dout, causal=causal)
    assert np.array_equal(a["o"], r["o"])
    assert np.array_equal(a["lse"], r["lse"])
    assert np.array_equal(a["dq"], r["dq"])
    dk_sum = r["dk"].reshape(B, T, Hkv, G, d).sum(axis=3)
    dv_sum = r["dv"].reshape(B, T, Hkv, G, d).sum(axis=3)
    np.testing.assert_allclose(a["dk"], dk_sum, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a["dv"], dv_sum, rtol=1e-12, atol=1e-13)
    # the forward entry point agrees with the backward's own O and LSE
    o, lse = oracle.fwd(q, k, v, causal=causal)
    assert np.array_equal(o, a["o"]) and np.array_equal(lse, a["lse"])


# ---------------------------------------------------------------- closed forms
def test_first_row_closed_form():
    B, T, Hq, Hkv, d = 2, 33, 4, 1, 16
    q, k, v, _ = rand_case(B, T, Hq, Hkv, d, seed=4, std=1.5)
    o, lse = oracle.fwd(q, k, v)
    for b in range(B):
        for h in range(Hq):
            assert np.allclose(o[b, 0, h], v[b, 0, 0], rtol=0, atol=1e-15)
            assert abs(lse[b, h, 0] - float(q[b, 0, h] @ k[b, 0, 0]) / math.sqrt(d)) <= 1e-14


@pytest.mark.parametrize("causal", [True, False])
def test_constant_keys_closed_form(causal):
    B, T, Hq, Hkv, d = 1, 29, 3, 1, 8
    rng = np.random.default_rng(8)
    q = rand((B, T, Hq, d), rng)
    k = np.ascontiguousarray(np.broadcast_to(rng.standard_normal((1, 1, 1, d)), (B, T, Hkv, d)))
    v = rand((B, T, Hkv, d), rng)
    o, lse = oracle.fwd(q, k, v, causal=causal)
    for i in range(T):
        n = i + 1 if causal else T
        mean_v = v[0, :n, 0].mean(axis=0)
        for h in range(Hq):
            s = float(q[0, i, h] @ k[0, 0, 0]) / math.sqrt(d)
            assert np.allclose(o[0, i, h], mean_v, rtol=0, atol=1e-13)
            assert abs(lse[0, h, i] - (s + math.log(n))) <= 1e-13


def test_single_token_gradients():
    B, T, Hq, Hkv, d = 2, 1, 6, 2, 8
    q, k, v, dout = rand_case(B, T, Hq, Hkv, d, seed=13)
    g = oracle.bwd(q, k, v, dout)
    assert np.allclose(g["dq"], 0, atol=1e-15)
    assert np.allclose(g["dk"], 0, atol=1e-15)
    expect_dv = dout.reshape(B, T, Hkv, Hq // Hkv, d).sum(axis=3)
    assert np.allclose(g["dv"], expect_dv, rtol=0, atol=1e-14)


# ---------------------------------------------------------------- hand-worked example
def _val(s):
    if isinstance(s, (int, float)):
        return float(s)
    env = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "ln6": math.log(6)}
    expr = s
    for key, val in env.items():
        expr = expr.replace(key, repr(val))
    # plain fractions and the logs above only
    return float(eval(expr, {"__builtins__": {}}, {"Fraction": Fraction}))


def test_worked_example_golden():
    with open(os.path.join(HERE, "golden", "worked_example_T3.json")) as f:
        gold = json.load(f)
    inp = {name: np.array([[_val(x) for x in row] for row in rows], dtype=np.float64)
           for name, rows in gold["inputs"].items()}
    q = inp["q"].reshape(1, 3, 1, 2)
    k = inp["k"].reshape(1, 3, 1, 2)
    v = inp["v"].reshape(1, 3, 1, 2)
    dout = inp["dO"].reshape(1, 3, 1, 2)
    g = oracle.bwd(q, k, v, dout, causal=True, scale=gold["shape"]["scale"])
    exp = gold["expected"]
    np.testing.assert_allclose(g["lse"].reshape(3), [_val(x) for x in exp["lse"]], rtol=0, atol=1e-15)
    for name in ("o", "dq", "dk", "dv"):
        want = np.array([[_val(x) for x in row] for row in exp[name]])
        np.testing.assert_allclose(g[name].reshape(3, 2), want, rtol=0, atol=1e-15, err_msg=name)


# ---------------------------------------------------------------- torch float64 special case
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(2, 17, 6, 2, 16), (1, 40, 4, 4, 8), (1, 9, 8, 1, 12)])
def test_against_torch_sdpa_f64(shape, causal):
    B, T, Hq, Hkv, d = shape
    q, k, v, dout = rand_case(B, T, Hq, Hkv, d, seed=17 + T)
    tq, tk, tv = (torch.tensor(x).transpose(1, 2).contiguous().requires_grad_(True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, enable_gqa=True)
    to.backward(torch.tensor(dout).transpose(1, 2))
    g = oracle.bwd(q, k, v, dout, causal=causal)
    tol = dict(rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["o"], to.detach().transpose(1, 2).numpy(), **tol)
    np.testing.assert_allclose(g["dq"], tq.grad.transpose(1, 2).numpy(), **tol)
    np.testing.assert_allclose(g["dk"], tk.grad.transpose(1, 2).numpy(), **tol)
    np.testing.assert_allclose(g["dv"], tv.grad.transpose(1, 2).numpy(), **tol)
    # LSE from torch's own logsumexp over the masked score matrix
    G = Hq // Hkv
    s = torch.einsum("bhid,bhjd->bhij", tq.detach(), tk.detach().repeat_interleave(G, dim=1)) / math.sqrt(d)
    if causal:
        s = s.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(g["lse"], torch.logsumexp(s, dim=-1).numpy(), **tol)


def test_bad_shapes_rejected():
    q, k, v, _ = rand_case(1, 4, 3, 2, 8, seed=1)  # 3 % 2 != 0
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v)


# ---------------------------------------------------------------- rotary embedding (oracle.rope)
def test_rope_closed_forms():
    """d = 2: one pair at frequency 1, so token t turns (1, 0) into (cos t, sin t); d = 4:
    the second pair turns at base**(-1/2) = 0.01 per token (1 radian at token 100); token 0
    is left as it is."""
    x = np.zeros((1, 101, 1, 2))
    x[..., 0] = 1.0
    y = oracle.rope(x)
    t = np.arange(101)
    np.testing.assert_allclose(y[0, :, 0, 0], np.cos(t), rtol=0, atol=1e-15)
    np.testing.assert_allclose(y[0, :, 0, 1], np.sin(t), rtol=0, atol=1e-15)
    x4 = np.zeros((1, 101, 1, 4))
    x4[..., 2] = 1.0
    y4 = oracle.rope(x4)
    assert abs(y4[0, 100, 0, 2] - math.cos(1.0)) < 1e-14 and abs(y4[0, 100, 0, 3] - math.sin(1.0)) < 1e-14
    assert np.all(y4[0, :, 0, :2] == 0.0)
    r = rand((2, 5, 3, 8), np.random.default_rng(3))
    assert np.array_equal(oracle.rope(r)[:, 0], r[:, 0])


def test_rope_preserves_pair_norms_and_inverts():
    x = rand((2, 40, 3, 16), np.random.default_rng(4))
    y = oracle.rope(x, base=500.0)
    n_x = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n_y = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(n_y, n_x, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.rope(y, base=500.0, inverse=True), x, rtol=0, atol=1e-13)


def test_rope_scores_depend_on_relative_position_only():
    """<rope(q) at m, rope(k) at n> is a function of m - n: shifting both by s keeps it."""
    rng = np.random.default_rng(5)
    d, T = 12, 64
    qv, kv = rng.standard_normal(d), rng.standard_normal(d)
    q = np.broadcast_to(qv, (1, T, 1, d)).copy()
    k = np.broadcast_to(kv, (1, T, 1, d)).copy()
    rq, rk = oracle.rope(q), oracle.rope(k)
    for m, n, s in ((10, 3, 17), (40, 40, 5), (2, 30, 20)):
        a = rq[0, m, 0] @ rk[0, n, 0]
        b = rq[0, m + s, 0] @ rk[0, n + s, 0]
        assert abs(a - b) < 1e-12, (m, n, s)


def test_rope_gradient_is_inverse_rotation():
    """Finite differences of L = sum(w * rope(x)) equal rope(w, inverse=True). The rotation
    is linear, so a central difference is exact for any step; a large one keeps the
    cancellation error near 1e-15."""
    rng = np.random.default_rng(6)
    x, w = rand((1, 9, 2, 6), rng), rand((1, 9, 2, 6), rng)
    g = oracle.rope(w, inverse=True)
    u = rand(x.shape, rng)
    u /= np.linalg.norm(u)
    eps = 0.25
    fd = (np.sum(w * oracle.rope(x + eps * u)) - np.sum(w * oracle.rope(x - eps * u))) / (2 * eps)
    assert abs(fd - np.sum(g * u)) < 1e-12
