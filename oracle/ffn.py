"""Plain fp64 CPU oracle for the blockwise feed-forward layer and its
gradients.

TEST INFRASTRUCTURE ONLY.  Nothing on the CUDA product path imports or calls
this module; it shares no code, header, table or helper with it.  Inputs are
the exact values handed to the GPU, upcast to float64.

Source (page title, section): "Ring Attention with Blockwise Transformers for
Near-Infinite Context" (arXiv 2310.01889 page), Abstract: the method computes
self-attention AND the feedforward network blockwise, and the blockwise
result is exact.  The feedforward is position-wise, so computing it one block
of tokens at a time changes only which hidden activations exist at once, not
the values: the plain definition below is the reference, and the blocked mode
must agree with it to rounding.

Readings where the pages are silent (each listed in the design notes): the
layer is the Transformer's position-wise feedforward y = act(x W1^T) W2^T with
hidden width 4 d_model and no biases; act is GELU in its exact form
GELU(u) = u Phi(u), Phi the standard normal CDF; the backward differentiates
L = sum(y * dy).

Layout: x, y, dy, dx are [T, d_model] (tokens of all batches flattened);
W1 is [d_hidden, d_model] and W2 is [d_model, d_hidden] (output x input, the
usual dense-layer layout).
"""
import math

import numpy as np

SQRT_HALF = 1.0 / math.sqrt(2.0)
INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)
_erf = np.vectorize(math.erf, otypes=[np.float64])


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def phi_cdf(u):
    """Standard normal CDF Phi(u) = (1 + erf(u / sqrt 2)) / 2."""
    return 0.5 * (1.0 + _erf(_f64(u) * SQRT_HALF))


def gelu(u):
    """GELU(u) = u Phi(u) (exact form, not the tanh approximation)."""
    u = _f64(u)
    return u * phi_cdf(u)


def gelu_grad(u):
    """d/du [u Phi(u)] = Phi(u) + u phi(u), phi the standard normal density."""
    u = _f64(u)
    return phi_cdf(u) + u * INV_SQRT_2PI * np.exp(-0.5 * u * u)


def ffn_fwd(x, w1, w2):
    """y = GELU(x W1^T) W2^T; also returns the pre-activation h = x W1^T."""
    x, w1, w2 = _f64(x), _f64(w1), _f64(w2)
    h = x @ w1.T
    return gelu(h) @ w2.T, h


def ffn_bwd(x, w1, w2, dy):
    """Gradients of L = sum(y * dy) by the chain rule:
    a = GELU(h), dA = dy W2, dH = dA * GELU'(h), dx = dH W1,
    dW2 = dy^T a, dW1 = dH^T x.  Returns (dx, dw1, dw2, y)."""
    x, w1, w2, dy = _f64(x), _f64(w1), _f64(w2), _f64(dy)
    h = x @ w1.T
    a = gelu(h)
    y = a @ w2.T
    dh = (dy @ w2) * gelu_grad(h)
    return dh @ w1, dh.T @ x, dy.T @ a, y


def ffn_blocked(x, w1, w2, block):
    """The forward one block of `block` tokens at a time, as the blockwise
    transformer computes it: only one block's hidden activations exist at a
    time; the outputs are concatenated."""
    x = _f64(x)
    out = [ffn_fwd(x[t:t + block], w1, w2)[0] for t in range(0, x.shape[0], block)]
    return np.concatenate(out, axis=0)


def ffn_bwd_blocked(x, w1, w2, dy, block):
    """The backward one block at a time: each block recomputes its hidden
    activations; dx is concatenated and the weight gradients are summed over
    blocks."""
    x, dy = _f64(x), _f64(dy)
    dxs, dw1, dw2 = [], 0.0, 0.0
    for t in range(0, x.shape[0], block):
        dx_b, dw1_b, dw2_b, _ = ffn_bwd(x[t:t + block], w1, w2, dy[t:t + block])
        dxs.append(dx_b)
        dw1 = dw1 + dw1_b
        dw2 = dw2 + dw2_b
    return np.concatenate(dxs, axis=0), dw1, dw2
