"""Pins of the oracle's attention half of a layer (oracle.layer_attn, oracle.rmsnorm),
which the whole-layer check of the GPU attention compares against.

As the page checks its model ("A transformer in PTX", §Checking the gradients):
awkward sizes (width 48, 4 query heads of 12 over 2 key/value heads, 3 sequences of
9 tokens), and for every parameter tensor the central difference of the loss along a
unit direction, once random and once along the gradient, against g . u. In f64 the
step can be small enough that the difference is exact to ~1e-8. Plus closed forms of
RMSNorm and the special case of a zero output projection."""
import numpy as np
import pytest

import oracle

B, T, C, HQ, HKV, D = 3, 9, 48, 4, 2, 12


def layer_inputs(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, T, C))
    g = 1.0 + 0.2 * rng.standard_normal(C)
    w_qkv = rng.standard_normal(((HQ + 2 * HKV) * D, C)) / np.sqrt(C)
    w_o = rng.standard_normal((C, HQ * D)) / np.sqrt(HQ * D)
    dx2 = rng.standard_normal((B, T, C))
    return rng, [x, g, w_qkv, w_o], dx2


@pytest.mark.parametrize("along", ["random", "gradient"])
def test_layer_gradients_match_central_differences(along):
    rng, params, dx2 = layer_inputs(7)
    out = oracle.layer_attn(*params, HQ, HKV, D, dx2)
    grads = [out["dx"], out["dg"], out["dw_qkv"], out["dw_o"]]
    for i, (p, gr) in enumerate(zip(params, grads)):
        u = rng.standard_normal(p.shape) if along == "random" else gr.copy()
        u /= np.linalg.norm(u)
        eps = 1e-5
        plus = [q if j != i else p + eps * u for j, q in enumerate(params)]
        minus = [q if j != i else p - eps * u for j, q in enumerate(params)]
        fd = (oracle.layer_attn_loss(*plus, HQ, HKV, D, dx2) - oracle.layer_attn_loss(*minus, HQ, HKV, D, dx2)) / (2 * eps)
        an = float(np.sum(gr * u))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(fd)), (i, fd, an)


def test_layer_forward_matches_its_loss_and_composition():
    _, params, dx2 = layer_inputs(8)
    out = oracle.layer_attn(*params, HQ, HKV, D, dx2)
    assert np.isclose(np.sum(out["x2"] * dx2), oracle.layer_attn_loss(*params, HQ, HKV, D, dx2), rtol=1e-12)
    # the attention output is the oracle's attention of the rotated projections
    o, _ = oracle.fwd(np.ascontiguousarray(oracle.rope(out["q"])), np.ascontiguousarray(oracle.rope(out["k"])),
                      np.ascontiguousarray(out["v"]))
    assert np.allclose(o, out["o"], rtol=0, atol=1e-12)


def test_zero_output_projection_passes_the_residual():
    """w_o = 0: x2 = x, dx = dx2, and nothing reaches the norm or the qkv weights."""
    _, (x, g, w_qkv, w_o), dx2 = layer_inputs(9)
    out = oracle.layer_attn(x, g, w_qkv, np.zeros_like(w_o), HQ, HKV, D, dx2)
    assert np.array_equal(out["x2"], x)
    assert np.allclose(out["dx"], dx2, rtol=0, atol=1e-15)
    assert np.max(np.abs(out["dg"])) == 0.0 and np.max(np.abs(out["dw_qkv"])) == 0.0


def test_rmsnorm_closed_forms():
    # a constant row c: mean(x^2) = c^2, so y = g c / sqrt(c^2 + eps)
    g = np.linspace(0.5, 1.5, 8)
    for c in (2.0, -0.25):
        y, r = oracle.rmsnorm(np.full((1, 8), c), g, eps=1e-5)
        assert np.allclose(y[0], g * c / np.sqrt(c * c + 1e-5), rtol=1e-15, atol=0)
        assert np.isclose(r[0], 1 / np.sqrt(c * c + 1e-5), rtol=1e-15)
    # with eps = 0 the output has root mean square |g|-weighted 1: sum((y/g)^2) / C = 1
    x = np.random.default_rng(3).standard_normal((4, 16))
    y, _ = oracle.rmsnorm(x, np.full(16, 2.0), eps=0.0)
    assert np.allclose(np.mean((y / 2.0) ** 2, axis=-1), 1.0, rtol=1e-14)


def test_rmsnorm_backward_matches_central_differences():
    rng = np.random.default_rng(4)
    x, g, dy = rng.standard_normal((2, 3, 10)), rng.standard_normal(10), rng.standard_normal((2, 3, 10))
    _, r = oracle.rmsnorm(x, g)
    dx, dg = oracle.rmsnorm_bwd(x, g, r, dy)
    loss = lambda xx, gg: float(np.sum(oracle.rmsnorm(xx, gg)[0] * dy))  # noqa: E731
    for _ in range(3):
        u = rng.standard_normal(x.shape)
        fd = (loss(x + 1e-6 * u, g) - loss(x - 1e-6 * u, g)) / 2e-6
        assert abs(fd - np.sum(dx * u)) <= 1e-7 * max(1, abs(fd))
        w = rng.standard_normal(g.shape)
        fd = (loss(x, g + 1e-6 * w) - loss(x, g - 1e-6 * w)) / 2e-6
        assert abs(fd - np.sum(dg * w)) <= 1e-7 * max(1, abs(fd))
