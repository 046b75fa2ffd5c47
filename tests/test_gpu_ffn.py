"""GPU parity of the blockwise feed-forward layer (forward and backward)
against the fp64 oracle.

Tolerances come from the arithmetic (standard floating-point error bounds),
since none is stated for this layer: the tensor cores multiply exact 16-bit
operands and accumulate in fp32, so the only roundings are (i) the hidden
activation GELU(h), GELU'(h) and dH rounded to the 16-bit operand type
(unit roundoff u = 2^-9 for bf16, 2^-12 for fp16) and (ii) fp32 accumulation
over K terms (at most K * 2^-24 relative to the sum of absolute products).
For an output z = sum_k p_k q_k the bound is therefore
    |z_gpu - z| <= (c u + K 2^-24) * sum_k |p_k q_k|
with c = 2 for y and dW2 (one rounded factor, with slack) and c = 4 for dx and
dW1 (dH carries two roundings), plus u_out |z| when the output itself is
stored in a 16-bit type.  The sums of absolute products are formed in fp64
from the oracle's exact intermediates."""
import os

import numpy as np
import pytest
import torch

os.environ.setdefault("RA_WAIT_TIMEOUT_MS", "3000")

import oracle  # noqa: E402
from tests._parity import f64  # noqa: E402

pytestmark = pytest.mark.gpu

U = {torch.bfloat16: 2.0 ** -9, torch.float16: 2.0 ** -12, torch.float32: 0.0}


@pytest.fixture(scope="module")
def ra():
    import blockwise_exact_attention_ra_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _within(name, got, want, bound):
    err = np.abs(np.asarray(got, dtype=np.float64) - want)
    worst = float((err - bound).max())
    assert worst <= 0.0, f"{name}: error exceeds its bound by {worst:.3e} (max err {err.max():.3e})"
    return float(err.max())


def _abs_sums(x, w1, w2, dy):
    """Sums of absolute products for y, dx, dW1, dW2 (fp64, exact intermediates)."""
    h = x @ w1.T
    a = oracle.gelu(h)
    dh = (dy @ w2) * oracle.gelu_grad(h)
    return (np.abs(a) @ np.abs(w2).T, np.abs(dh) @ np.abs(w1), np.abs(dh).T @ np.abs(x),
            np.abs(dy).T @ np.abs(a))


def _case(ra, T, dm, dh, block, dtype, seed, out_dtype=torch.float32):
    from blockwise_exact_attention_ra_gb300.inputs import make_ffn
    x, w1, w2, dy = make_ffn(T, dm, dh, dtype, "cuda", seed)
    y = ra.ffn_fwd(x, w1, w2, block, y_dtype=out_dtype)
    dx, dw1, dw2 = ra.ffn_bwd(x, w1, w2, dy, block, dx_dtype=out_dtype)
    ra.ra_sync_status(None)
    X, W1, W2, DY = f64(x), f64(w1), f64(w2), f64(dy)
    rdx, rdw1, rdw2, ry = oracle.ffn_bwd(X, W1, W2, DY)
    sy, sdx, sdw1, sdw2 = _abs_sums(X, W1, W2, DY)
    u, uo = U[dtype], U[out_dtype]
    _within("y", f64(y), ry, (2 * u + dh * 2.0 ** -24) * sy + uo * np.abs(ry) + 1e-6)
    _within("dx", f64(dx), rdx, (4 * u + dh * 2.0 ** -24) * sdx + uo * np.abs(rdx) + 1e-6)
    _within("dW1", f64(dw1), rdw1, (4 * u + T * 2.0 ** -24) * sdw1 + 1e-6)
    _within("dW2", f64(dw2), rdw2, (2 * u + T * 2.0 ** -24) * sdw2 + 1e-6)
    return x, w1, w2, dy, y, dx, dw1, dw2


def test_ffn_bf16_one_block(ra):
    _case(ra, 256, 256, 1024, 256, torch.bfloat16, 501)


def test_ffn_bf16_several_blocks_ragged_tail(ra):
    # blocks of 256, 256 and 128 tokens; several 128 x 256 tiles in every product
    _case(ra, 640, 512, 2048, 256, torch.bfloat16, 502)


def test_ffn_fp16_operands_bf16_outputs(ra):
    _case(ra, 384, 256, 768, 128, torch.float16, 503, out_dtype=torch.bfloat16)


def test_ffn_block_size_does_not_change_the_result(ra):
    from blockwise_exact_attention_ra_gb300.inputs import make_ffn
    x, w1, w2, dy = make_ffn(1024, 512, 1024, torch.bfloat16, "cuda", 504)
    ys = [ra.ffn_fwd(x, w1, w2, b) for b in (128, 384, 1024)]
    gs = [ra.ffn_bwd(x, w1, w2, dy, b) for b in (128, 384, 1024)]
    ra.ra_sync_status(None)
    # each token's row of y and dx is computed by the same products whatever the block
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
    for g in gs[1:]:
        assert torch.equal(g[0], gs[0][0])
        # weight gradients: the same terms, summed in another grouping
        for a, b in ((g[1], gs[0][1]), (g[2], gs[0][2])):
            tol = 1e-5 * float(b.abs().max())
            assert float((a - b).abs().max()) <= tol


def test_ffn_bench_size_sampled(ra):
    # the bench workload's shape (131072 tokens, d_model 2048, hidden 8192, blocks
    # of 16384): rows of y and dx checked one by one, and sampled entries of dW1, dW2
    from blockwise_exact_attention_ra_gb300.inputs import make_ffn
    T, dm, dh, block = 131072, 2048, 8192, 16384
    x, w1, w2, dy = make_ffn(T, dm, dh, torch.bfloat16, "cuda", 505)
    y = ra.ffn_fwd(x, w1, w2, block, y_dtype=torch.float32)
    dx, dw1, dw2 = ra.ffn_bwd(x, w1, w2, dy, block)
    ra.ra_sync_status(None)
    rng = np.random.default_rng(7)
    rows = np.unique(np.r_[0, T - 1, block - 1, block, rng.integers(0, T, 60)])
    W1, W2 = f64(w1), f64(w2)
    X, DY = f64(x[rows]), f64(dy[rows])
    rdx, _, _, ry = oracle.ffn_bwd(X, W1, W2, DY)
    sy, sdx, _, _ = _abs_sums(X, W1, W2, DY)
    u = U[torch.bfloat16]
    _within("y rows", f64(y[rows]), ry, (2 * u + dh * 2.0 ** -24) * sy + 1e-6)
    _within("dx rows", f64(dx[rows]), rdx, (4 * u + dh * 2.0 ** -24) * sdx + 1e-6)
    # dW2[o, j] = sum_t dy[t, o] GELU(h[t, j]),  dW1[j, i] = sum_t dH[t, j] x[t, i]
    js = rng.integers(0, dh, 3)
    Xall = f64(x)
    DYall = f64(dy)
    for j in js:
        h = Xall @ W1[j]
        a = oracle.gelu(h)
        dHj = (DYall @ W2[:, j]) * oracle.gelu_grad(h)
        os_ = rng.integers(0, dm, 4)
        for o in os_:
            want = float(DYall[:, o] @ a)
            bound = (2 * u + T * 2.0 ** -24) * float(np.abs(DYall[:, o]) @ np.abs(a)) + 1e-6
            assert abs(float(dw2[o, j]) - want) <= bound, ("dW2", o, j)
            want1 = float(dHj @ Xall[:, o])
            bound1 = (4 * u + T * 2.0 ** -24) * float(np.abs(dHj) @ np.abs(Xall[:, o])) + 1e-6
            assert abs(float(dw1[j, o]) - want1) <= bound1, ("dW1", j, o)
