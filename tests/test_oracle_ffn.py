"""Pins for the fp64 feed-forward oracle, independent of its own formulas:
closed forms and identities of GELU, brute-force finite differences, torch's
exact GELU with autograd on tiny inputs, and planted mistakes (the tanh
approximation, a transposed weight, a dropped derivative factor) that these
pins must catch."""
import math

import numpy as np
import pytest

import oracle
from oracle import ffn as F

RNG = np.random.default_rng(20260514)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def test_gelu_closed_forms():
    assert F.gelu(0.0) == 0.0
    # Phi(0) = 1/2, so GELU'(0) = 1/2
    assert abs(F.gelu_grad(0.0) - 0.5) < 1e-15
    # far tails: GELU(u) -> u for u >> 0 and -> 0 for u << 0
    assert abs(F.gelu(40.0) - 40.0) < 1e-12 and abs(F.gelu(-40.0)) < 1e-12
    # Phi(1) from the normal table: 0.8413447460685429
    assert abs(F.gelu(1.0) - 0.8413447460685429) < 1e-15


def test_gelu_odd_part_is_identity():
    # Phi(u) + Phi(-u) = 1  =>  GELU(u) - GELU(-u) = u for every u
    u = rand(1000, scale=3.0)
    np.testing.assert_allclose(F.gelu(u) - F.gelu(-u), u, atol=1e-14)


def test_gelu_grad_is_the_derivative():
    u = rand(200, scale=2.0)
    eps = 1e-6
    fd = (F.gelu(u + eps) - F.gelu(u - eps)) / (2 * eps)
    np.testing.assert_allclose(F.gelu_grad(u), fd, rtol=1e-8, atol=1e-9)


def test_ffn_matches_torch_exact_gelu_with_autograd():
    torch = pytest.importorskip("torch")
    T, dm, dh = 7, 5, 12
    x, w1, w2, dy = rand(T, dm), rand(dh, dm), rand(dm, dh), rand(T, dm)
    tx, t1, t2 = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (x, w1, w2))
    ty = torch.nn.functional.linear(torch.nn.functional.gelu(torch.nn.functional.linear(tx, t1)), t2)
    ty.backward(torch.tensor(dy))
    dx, dw1, dw2, y = oracle.ffn_bwd(x, w1, w2, dy)
    np.testing.assert_allclose(y, ty.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(oracle.ffn_fwd(x, w1, w2)[0], ty.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dx, tx.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dw1, t1.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dw2, t2.grad.numpy(), atol=1e-12)


def test_ffn_gradients_by_finite_differences():
    T, dm, dh = 4, 3, 6
    x, w1, w2, dy = rand(T, dm), rand(dh, dm), rand(dm, dh), rand(T, dm)
    dx, dw1, dw2, _ = oracle.ffn_bwd(x, w1, w2, dy)
    eps = 1e-6

    def loss(x_, w1_, w2_):
        return float((oracle.ffn_fwd(x_, w1_, w2_)[0] * dy).sum())

    for name, arr, grad in (("x", x, dx), ("w1", w1, dw1), ("w2", w2, dw2)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = [p if n == name else a for n, a in (("x", x), ("w1", w1), ("w2", w2))]
            args_m = [m if n == name else a for n, a in (("x", x), ("w1", w1), ("w2", w2))]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-7, err_msg=name)


@pytest.mark.parametrize("block", [1, 2, 3, 8])
def test_blockwise_equals_whole(block):
    T, dm, dh = 8, 4, 16
    x, w1, w2, dy = rand(T, dm), rand(dh, dm), rand(dm, dh), rand(T, dm)
    np.testing.assert_allclose(oracle.ffn_blocked(x, w1, w2, block), oracle.ffn_fwd(x, w1, w2)[0], atol=1e-13)
    dxb, dw1b, dw2b = oracle.ffn_bwd_blocked(x, w1, w2, dy, block)
    dx, dw1, dw2, _ = oracle.ffn_bwd(x, w1, w2, dy)
    for got, want in ((dxb, dx), (dw1b, dw1), (dw2b, dw2)):
        np.testing.assert_allclose(got, want, atol=1e-12)


def test_position_wise_rows_are_independent():
    # each output row depends on its own input row only
    T, dm, dh = 6, 4, 8
    x, w1, w2 = rand(T, dm), rand(dh, dm), rand(dm, dh)
    y = oracle.ffn_fwd(x, w1, w2)[0]
    x2 = x.copy()
    x2[3] += 5.0
    y2 = oracle.ffn_fwd(x2, w1, w2)[0]
    assert np.array_equal(np.delete(y, 3, 0), np.delete(y2, 3, 0))
    assert not np.allclose(y[3], y2[3])


# --- planted mistakes: each must fail a pin above ------------------------------

def _tanh_gelu(u):
    u = np.asarray(u, dtype=np.float64)
    return 0.5 * u * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (u + 0.044715 * u ** 3)))


def test_planted_tanh_approximation_is_caught():
    u = np.linspace(-4, 4, 101)
    assert np.abs(_tanh_gelu(u) - F.gelu(u)).max() > 1e-5   # fails the torch exact-GELU pin


def test_planted_transposed_weight_is_caught():
    T, d = 5, 6   # square so the transposed weight still fits
    x, w1, w2 = rand(T, d), rand(d, d), rand(d, d)
    y = oracle.ffn_fwd(x, w1, w2)[0]
    bad = F.gelu(x @ w1) @ w2.T
    assert np.abs(bad - y).max() > 1e-3


def test_planted_dropped_derivative_factor_is_caught():
    T, dm, dh = 4, 3, 6
    x, w1, w2, dy = rand(T, dm), rand(dh, dm), rand(dm, dh), rand(T, dm)
    dx = oracle.ffn_bwd(x, w1, w2, dy)[0]
    bad = (dy @ w2) @ w1   # GELU'(h) left out
    assert np.abs(bad - dx).max() > 1e-3
