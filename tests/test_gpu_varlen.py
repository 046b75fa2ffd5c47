"""GPU parity of the ring with variable per-host lengths (dynamic masking):
host i's first len_i rows are its tokens, the rest is padding filled with
large garbage.  The oracle computes exact attention over the concatenated
valid rows; padded rows must come out as O = 0, LSE = -inf and zero
gradients, whatever the padding holds."""
import os

import numpy as np
import pytest
import torch

os.environ.setdefault("RA_WAIT_TIMEOUT_MS", "3000")

import oracle  # noqa: E402
from tests._parity import check, f64  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import blockwise_exact_attention_ra_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _varlen_case(ra, B, N, Hq, Hkv, d, P, lens, causal, dtype, seed, precise=False):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    q, k, v, do = make_tensors(B, N, Hq, Hkv, d, dtype, "cuda", seed)
    rows = torch.as_tensor(oracle.varlen_rows(N, P, lens), device="cuda")
    pad = torch.ones(N, dtype=torch.bool, device="cuda")
    pad[rows] = False
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    for t in (q, k, v, do):   # garbage in the padding (finite, inside fp16 range)
        t[:, pad] = (300.0 * torch.randn(t[:, pad].shape, generator=g, device="cuda")).to(dtype)
    hl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = d ** -0.5
    o, lse = ra.ring_attention_fwd(q, k, v, P, causal, scale, precise=precise, host_len=hl)
    dq, dk, dv = ra.ring_attention_bwd(q, k, v, o, lse, do, P, causal, scale, precise=precise, host_len=hl)
    ra.ra_sync_status()
    rq, rk, rv, rO, rL = oracle.attention_varlen(f64(q), f64(k), f64(v), f64(do), P, lens, causal, scale)
    check("varlen O", f64(o), rO, dtype)
    check("varlen LSE", f64(lse), rL, dtype, kind="lse")
    check("varlen dQ", f64(dq), rq, dtype)
    check("varlen dK", f64(dk), rk, dtype)
    check("varlen dV", f64(dv), rv, dtype)


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_tc_ragged_hosts(ra, causal):
    # full, partial tile, empty, exactly one tile, several partial tiles
    _varlen_case(ra, 1, 5 * 512, 2, 2, 128, 5, [512, 77, 0, 128, 300], causal, torch.bfloat16, 71)


def test_varlen_tc_gqa_two_batches(ra):
    _varlen_case(ra, 2, 4 * 384, 4, 2, 128, 4, [384, 1, 256, 129], True, torch.bfloat16, 72)


def test_varlen_tc_head_dim_64_precise(ra):
    _varlen_case(ra, 1, 3 * 256, 2, 1, 64, 3, [200, 256, 5], True, torch.bfloat16, 73, precise=True)


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_all_hosts_empty(ra, causal):
    # every row is padding: O = 0, LSE = -inf, zero gradients, no tile visited
    _varlen_case(ra, 1, 4 * 128, 2, 2, 128, 4, [0, 0, 0, 0], causal, torch.bfloat16, 75)
    _varlen_case(ra, 1, 4 * 64, 2, 2, 64, 4, [0, 0, 0, 0], causal, torch.float32, 76)


def test_varlen_fp32(ra):
    _varlen_case(ra, 1, 4 * 64, 2, 2, 64, 4, [64, 10, 0, 33], True, torch.float32, 74)


def test_varlen_full_lengths_equal_plain_ring(ra):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    q, k, v, do = make_tensors(1, 1024, 2, 2, 128, torch.bfloat16, "cuda", 75)
    hl = torch.full((4,), 256, dtype=torch.int32, device="cuda")
    o1, l1 = ra.ring_attention_fwd(q, k, v, 4, True)
    o2, l2 = ra.ring_attention_fwd(q, k, v, 4, True, host_len=hl)
    g1 = ra.ring_attention_bwd(q, k, v, o1, l1, do, 4, True)
    g2 = ra.ring_attention_bwd(q, k, v, o2, l2, do, 4, True, host_len=hl)
    ra.ra_sync_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
