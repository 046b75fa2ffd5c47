"""bench.py accounting: the per-row flops used for the CPU baseline add up to
the whole-problem formula used for the GPU metric, and the formula matches the
stated causal-adjusted counts (fwd 4*B*H*N^2*d/2, bwd 2.5x fwd)."""
import pytest

import bench


def test_causal_flops_formula():
    fwd, bwd = bench.algo_flops(1, 131072, 16, 128, causal=True)
    assert fwd == pytest.approx(70.37e12, rel=1e-3)
    assert bwd == pytest.approx(175.9e12, rel=1e-3)
    fwd_nc, _ = bench.algo_flops(1, 512, 2, 64, causal=False)
    assert fwd_nc == 4 * 2 * 512 * 512 * 64


@pytest.mark.parametrize("N,H,d", [(64, 3, 32), (1024, 2, 128)])
def test_row_flops_sum_to_whole_problem(N, H, d):
    fwd, bwd = bench.algo_flops(1, N, H, d, causal=True)
    rows = H * sum(bench.row_flops(i, d, True, N) for i in range(N))
    # rows see i+1 keys: N(N+1)/2 visible pairs against the formula's N^2/2
    assert rows == pytest.approx((fwd + bwd) * (N + 1) / N, rel=1e-12)
    rows_nc = H * sum(bench.row_flops(i, d, False, N) for i in range(N))
    f2, b2 = bench.algo_flops(1, N, H, d, causal=False)
    assert rows_nc == pytest.approx(f2 + b2, rel=1e-12)
