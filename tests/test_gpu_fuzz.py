"""Seeded random sweep over the ring's parameter space: each case draws the
batch, head counts and grouping, head dimension, number of hosts, host block
size, mask, operand type, layout (contiguous, striped or variable host
lengths) and memory order of the tensors ([B, N, H, d] rows or [B, H, N, d]
heads, passed as strides), runs the ring forward and backward on the GPU and
compares every output with the fp64 oracle at the stated tolerances.  The draws are fixed by
the seed, so the sweep is the same on every run."""
import os

import numpy as np
import pytest
import torch

os.environ.setdefault("RA_WAIT_TIMEOUT_MS", "3000")

import oracle  # noqa: E402
from tests._parity import check, f64  # noqa: E402

pytestmark = pytest.mark.gpu


def _draw(n, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        B = int(rng.choice([1, 2]))
        Hkv = int(rng.choice([1, 2]))
        group = int(rng.choice([1, 2, 4]))
        d = int(rng.choice([64, 128]))
        P = int(rng.choice([1, 2, 3, 4]))
        S = int(rng.choice([128, 256]))
        causal = bool(rng.random() < 0.7)
        dtype = "bf16" if rng.random() < 0.7 else "fp16"
        layout = rng.choice(["contiguous", "striped", "varlen"]) if causal else rng.choice(["contiguous", "varlen"])
        lens = [int(x) for x in rng.integers(0, S + 1, P)]
        if layout == "varlen" and sum(lens) == 0:
            lens[0] = S
        order = "heads" if rng.random() < 0.3 else "rows"
        cases.append(dict(B=B, Hkv=Hkv, Hq=Hkv * group, d=d, P=P, S=S, causal=causal, dtype=dtype,
                          layout=str(layout), lens=lens, order=order, seed=900 + i))
    return cases


CASES = _draw(24)


@pytest.fixture(scope="module")
def ra():
    import blockwise_exact_attention_ra_gb300 as ra
    assert torch.cuda.is_available()
    return ra


@pytest.mark.parametrize("c", CASES, ids=[f"{c['layout']}-B{c['B']}-Hq{c['Hq']}-Hkv{c['Hkv']}-d{c['d']}-P{c['P']}-S{c['S']}-"
                                          f"{'causal' if c['causal'] else 'full'}-{c['dtype']}-{c['order']}" for c in CASES])
def test_random_ring_case(ra, c):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    dtype = torch.bfloat16 if c["dtype"] == "bf16" else torch.float16
    B, Hq, Hkv, d, P, S = c["B"], c["Hq"], c["Hkv"], c["d"], c["P"], c["S"]
    N = P * S
    q, k, v, do = make_tensors(B, N, Hq, Hkv, d, dtype, "cuda", c["seed"])
    scale = d ** -0.5

    def order(t):  # the same values in [B, H, N, d] memory order when drawn
        return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) if c["order"] == "heads" else t
    if c["layout"] == "striped":
        pos = torch.as_tensor(oracle.striped_positions(N, P), device="cuda")
        inv = torch.argsort(pos)
        qs, ks, vs, dos = (order(t[:, pos].contiguous()) for t in (q, k, v, do))
        o, lse = ra.ring_attention_fwd(qs, ks, vs, P, True, scale, striped=True)
        dq, dk, dv = ra.ring_attention_bwd(qs, ks, vs, o, lse, dos, P, True, scale, striped=True)
        ra.ra_sync_status()
        o, lse, dq, dk, dv = o[:, inv], lse[:, :, inv], dq[:, inv], dk[:, inv], dv[:, inv]
        rq, rk, rv, rO, rL, _ = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), True, scale)
    elif c["layout"] == "varlen":
        hl = torch.tensor(c["lens"], dtype=torch.int32, device="cuda")
        qo, ko, vo, doo = (order(t) for t in (q, k, v, do))
        o, lse = ra.ring_attention_fwd(qo, ko, vo, P, c["causal"], scale, host_len=hl)
        dq, dk, dv = ra.ring_attention_bwd(qo, ko, vo, o, lse, doo, P, c["causal"], scale, host_len=hl)
        ra.ra_sync_status()
        rq, rk, rv, rO, rL = oracle.attention_varlen(f64(q), f64(k), f64(v), f64(do), P, c["lens"], c["causal"],
                                                     scale)
    else:
        qo, ko, vo, doo = (order(t) for t in (q, k, v, do))
        o, lse = ra.ring_attention_fwd(qo, ko, vo, P, c["causal"], scale)
        dq, dk, dv = ra.ring_attention_bwd(qo, ko, vo, o, lse, doo, P, c["causal"], scale)
        ra.ra_sync_status()
        rq, rk, rv, rO, rL, _ = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), c["causal"], scale)
    check("O", f64(o), rO, dtype)
    check("LSE", f64(lse), rL, dtype, kind="lse")
    check("dQ", f64(dq), rq, dtype)
    check("dK", f64(dk), rk, dtype)
    check("dV", f64(dv), rv, dtype)
