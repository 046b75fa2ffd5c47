"""GPU parity at the named workloads' ring structure, element by element.

The named workloads run 32 or 64 virtual hosts with host blocks of 4096 to
16384 rows; at their full sizes the fp64 oracle can only check sampled rows.
These cases keep that structure -- many hosts, many query tiles per host, more
key/value tiles than the GPU has SMs, so the backward's schedule runs several
rounds -- at lengths where the oracle computes every output, and compare
O, LSE, dQ, dK and dV in full.

They also check what the pages' "What I Still Don't Understand" section
raises: a small loss gap that its author puts down to floating-point error
piling up over ring steps.  Here the same seeded inputs run with P = 1, 4, 16
and 64 hosts; every P must meet the tolerance, the largest error at P = 64
must stay within twice that at P = 1, and under a causal mask the kernels
visit every query tile's key tiles in the same order for every P, so O, LSE,
dK and dV must not change at all.
"""
import os

import numpy as np
import pytest
import torch

os.environ.setdefault("RA_WAIT_TIMEOUT_MS", "3000")

import oracle  # noqa: E402
from tests._parity import TOL, check, f64  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import blockwise_exact_attention_ra_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _inputs(N, Hq, Hkv, seed, d=128, dtype=torch.bfloat16):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    return make_tensors(1, N, Hq, Hkv, d, dtype, "cuda", seed)


def _oracle(q, k, v, do, causal, scale):
    return oracle.attention_bwd_by_row_blocks(f64(q), f64(k), f64(v), f64(do), causal, scale)


def _check_all(tag, got, want, dtype=torch.bfloat16):
    o, lse, dq, dk, dv = got
    errs = {}
    errs["O"] = check(f"{tag} O", f64(o), want["O"], dtype)
    errs["LSE"] = check(f"{tag} LSE", f64(lse), want["LSE"], dtype, kind="lse")
    errs["dQ"] = check(f"{tag} dQ", f64(dq), want["dQ"], dtype)
    errs["dK"] = check(f"{tag} dK", f64(dk), want["dK"], dtype)
    errs["dV"] = check(f"{tag} dV", f64(dv), want["dV"], dtype)
    return errs


def _run(ra, q, k, v, do, P, causal, scale, **kw):
    o, lse = ra.ring_attention_fwd(q, k, v, P, causal, scale, **kw)
    dq, dk, dv = ra.ring_attention_bwd(q, k, v, o, lse, do, P, causal, scale, **kw)
    ra.ra_sync_status()
    return o, lse, dq, dk, dv


# (N, Hq, Hkv, P, causal): S = N / P rows per host
STRUCTURES = [
    (4096, 2, 2, 32, True),     # 32 hosts of one 128-row tile (the bench's host count)
    (8192, 1, 1, 64, True),     # 64 hosts of one tile (the 1M-token workload's host count)
    (8192, 1, 1, 64, False),    # the same without a mask: every host wraps around the ring
    (8192, 4, 1, 32, True),     # 32 hosts of two tiles, four query heads per key/value head
    (32768, 2, 2, 8, True),     # hosts of 4096 rows (the bench's host size), 512 key tiles
]


@pytest.mark.parametrize("N,Hq,Hkv,P,causal", STRUCTURES,
                         ids=[f"N{s[0]}-Hq{s[1]}-Hkv{s[2]}-P{s[3]}-{'causal' if s[4] else 'full'}"
                              for s in STRUCTURES])
def test_full_gradients_at_ring_structure(ra, N, Hq, Hkv, P, causal):
    q, k, v, do = _inputs(N, Hq, Hkv, 3000 + N // 1024 + P + Hq)
    scale = 128 ** -0.5
    got = _run(ra, q, k, v, do, P, causal, scale)
    _check_all(f"N{N} P{P}", got, _oracle(q, k, v, do, causal, scale))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_full_gradients_two_batches_head_dim_64_32_hosts(ra, dtype):
    # two batches (batch strides), d = 64 and fp16 inputs at 32 hosts of 128 rows
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    N, P = 4096, 32
    q, k, v, do = make_tensors(2, N, 4, 2, 64, dtype, "cuda", 3050 + int(dtype == torch.float16))
    scale = 64 ** -0.5
    got = _run(ra, q, k, v, do, P, True, scale)
    _check_all(f"B2 d64 {dtype} P{P}", got, _oracle(q, k, v, do, True, scale), dtype)


def test_striped_full_gradients_32_hosts(ra):
    N, H, P = 4096, 2, 32
    q, k, v, do = _inputs(N, H, H, 3101)
    scale = 128 ** -0.5
    pos = torch.as_tensor(oracle.striped_positions(N, P), device="cuda")
    inv = torch.argsort(pos)
    qs, ks, vs, dos = (t[:, pos].contiguous() for t in (q, k, v, do))
    o, lse, dq, dk, dv = _run(ra, qs, ks, vs, dos, P, True, scale, striped=True)
    got = (o[:, inv], lse[:, :, inv], dq[:, inv], dk[:, inv], dv[:, inv])
    _check_all("striped P32", got, _oracle(q, k, v, do, True, scale))


def test_variable_lengths_full_gradients_32_hosts(ra):
    N, H, P = 8192, 2, 32
    S = N // P
    q, k, v, do = _inputs(N, H, H, 3102)
    scale = 128 ** -0.5
    rng = np.random.default_rng(3102)
    lens = [int(x) for x in rng.integers(0, S + 1, P)]
    lens[0], lens[5], lens[17] = S, 0, 1   # a full host, an empty host, a single token
    hl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    got = _run(ra, q, k, v, do, P, True, scale, host_len=hl)
    rq, rk, rv, rO, rL = oracle.attention_varlen(f64(q), f64(k), f64(v), f64(do), P, lens, True, scale)
    _check_all("varlen P32", got, {"O": rO, "LSE": rL, "dQ": rq, "dK": rk, "dV": rv})


@pytest.mark.parametrize("causal", [True, False])
def test_error_does_not_grow_with_host_count(ra, causal):
    N, H = 8192, 2
    q, k, v, do = _inputs(N, H, H, 3200 + int(causal))
    scale = 128 ** -0.5
    want = _oracle(q, k, v, do, causal, scale)
    errs, outs = {}, {}
    for P in (1, 4, 16, 64):
        got = _run(ra, q, k, v, do, P, causal, scale)
        errs[P] = _check_all(f"P{P}", got, want)
        outs[P] = got
    for name in ("O", "LSE", "dQ", "dK", "dV"):
        floor = TOL[torch.bfloat16]["lse" if name == "LSE" else "max"] * 1e-3
        assert errs[64][name] <= 2.0 * max(errs[1][name], floor), (
            f"{name}: max |err| {errs[64][name]:.3e} at P=64 vs {errs[1][name]:.3e} at P=1")
    if causal:
        # same key-tile order for every query tile whatever P is: identical results
        # (dQ is summed by reduce-adds whose order varies from run to run)
        for P in (4, 16, 64):
            for i, name in ((0, "O"), (1, "LSE"), (3, "dK"), (4, "dV")):
                assert torch.equal(outs[P][i], outs[1][i]), f"{name} differs between P=1 and P={P}"


def test_backward_repeats_bitwise_except_dq(ra):
    N, H, P = 4096, 2, 32
    q, k, v, do = _inputs(N, H, H, 3300)
    scale = 128 ** -0.5
    o, lse = ra.ring_attention_fwd(q, k, v, P, True, scale)
    g1 = ra.ring_attention_bwd(q, k, v, o, lse, do, P, True, scale)
    g2 = ra.ring_attention_bwd(q, k, v, o, lse, do, P, True, scale)
    ra.ra_sync_status()
    assert torch.equal(g1[1], g2[1]), "dK differs between two runs"
    assert torch.equal(g1[2], g2[2]), "dV differs between two runs"
    # dQ: fp32 sums in a run-dependent order; the difference is rounding only
    diff = (g1[0] - g2[0]).abs().max().item()
    assert diff <= 1e-5 * max(1.0, g1[0].abs().max().item()), f"dQ runs differ by {diff:.3e}"
