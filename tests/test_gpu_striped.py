"""GPU parity of the striped (load-balanced) causal ring: inputs in the
original order are permuted to the striped layout (host i's local row l holds
position l*P + i), run through ra_ring_fwd / ra_ring_bwd with RA_STRIPED, and
the outputs, mapped back to the original order, are compared with the fp64
oracle on the original order."""
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


def _striped_case(ra, B, N, Hq, Hkv, d, P, dtype, seed, q_scale=1.0, outliers=0.0, precise=False):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    q, k, v, do = make_tensors(B, N, Hq, Hkv, d, dtype, "cuda", seed, q_scale, outliers)
    pos = torch.as_tensor(oracle.striped_positions(N, P), device="cuda")
    inv = torch.argsort(pos)
    scale = d ** -0.5
    qs, ks, vs, dos = (t[:, pos].contiguous() for t in (q, k, v, do))
    o, lse = ra.ring_attention_fwd(qs, ks, vs, P, True, scale, precise=precise, striped=True)
    dq, dk, dv = ra.ring_attention_bwd(qs, ks, vs, o, lse, dos, P, True, scale, precise=precise, striped=True)
    ra.ra_sync_status()
    rq, rk, rv, rO, rL, _ = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), True, scale)
    check("striped O", f64(o[:, inv]), rO, dtype)
    check("striped LSE", f64(lse[:, :, inv]), rL, dtype, kind="lse")
    check("striped dQ", f64(dq[:, inv]), rq, dtype)
    check("striped dK", f64(dk[:, inv]), rk, dtype)
    check("striped dV", f64(dv[:, inv]), rv, dtype)


@pytest.mark.parametrize("P", [1, 2, 4])
def test_striped_tc_bf16(ra, P):
    _striped_case(ra, 2, 1024, 2, 2, 128, P, torch.bfloat16, 61 + P)


def test_striped_tc_gqa_odd_tiles(ra):
    _striped_case(ra, 1, 1152, 4, 2, 128, 3, torch.bfloat16, 65)


def test_striped_tc_head_dim_64_precise_stress(ra):
    _striped_case(ra, 1, 1024, 2, 1, 64, 4, torch.bfloat16, 66, q_scale=4.0, outliers=0.01, precise=True)


def test_striped_fp32(ra):
    _striped_case(ra, 1, 512, 2, 1, 64, 4, torch.float32, 67)


def test_striped_equals_contiguous_when_one_host(ra):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    q, k, v, _ = make_tensors(1, 512, 2, 2, 128, torch.bfloat16, "cuda", 68)
    o1, l1 = ra.ring_attention_fwd(q, k, v, 1, True)
    o2, l2 = ra.ring_attention_fwd(q, k, v, 1, True, striped=True)
    ra.ra_sync_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
