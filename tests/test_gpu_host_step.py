"""GPU checks of ra_ring_step_host, the forward + backward step on tensors
in host memory.  It runs the kernels of ra_ring_fwd and ra_ring_bwd on device
copies of its inputs, so its outputs must equal theirs bit for bit whatever
the host memory (pinned or pageable), the batch strides of the host tensors
or the interleaving of calls on two streams; one fp32 case also goes to the
oracle."""
import os

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


def _device_step(ra, q, k, v, do, P, causal, scale, o_dtype, g_dtype, precise=False, striped=False):
    o, lse = ra.ring_attention_fwd(q, k, v, P, causal, scale, o_dtype=o_dtype, precise=precise,
                                   striped=striped)
    dq, dk, dv = ra.ring_attention_bwd(q, k, v, o, lse, do, P, causal, scale, grad_dtype=g_dtype,
                                       precise=precise, striped=striped)
    torch.cuda.synchronize()
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


def _host_tensor(t, pin, pad_rows=0):
    """Host copy of device tensor t; with pad_rows, a view into a larger
    buffer so the batch stride exceeds one batch."""
    B, N = t.shape[:2]
    if pad_rows:
        big = torch.zeros((B, N + pad_rows) + tuple(t.shape[2:]), dtype=t.dtype, pin_memory=pin)
        view = big[:, :N]
        view.copy_(t.cpu())
        return view
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=pin)
    h.copy_(t.cpu())
    return h


def _host_outputs(B, N, Hq, Hkv, d, o_dtype, g_dtype, pin, pad_rows=0):
    def buf(H, dt):
        if pad_rows:
            return torch.full((B, N + pad_rows, H, d), 7.0, dtype=dt, pin_memory=pin)[:, :N]
        return torch.full((B, N, H, d), 7.0, dtype=dt, pin_memory=pin)
    return [buf(Hq, o_dtype), torch.full((B, Hq, N), 7.0, dtype=torch.float32, pin_memory=pin),
            buf(Hq, g_dtype), buf(Hkv, g_dtype), buf(Hkv, g_dtype)]


def _run_host(ra, hin, hout, P, causal, scale, ws=None, stream=None, precise=False, striped=False):
    q, k = hin[0], hin[1]
    if ws is None:
        sh = ra.shape_of(q, k)
        nbytes = ra.ra_ring_step_host_workspace_bytes(ra._dt(q), ra._dt(hout[0]), ra._dt(hout[2]), sh, P)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ra.ra_ring_step_host(*hin, P, causal, scale, *hout, ws, stream, precise, striped)
    (stream or torch.cuda.current_stream()).synchronize()
    ra.ra_sync_status(stream)


def _case(ra, B, N, Hq, Hkv, d, P, causal, dtype, o_dtype, g_dtype, seed, pin=True, pad=0, **kw):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    q, k, v, do = make_tensors(B, N, Hq, Hkv, d, dtype, "cuda", seed)
    scale = d ** -0.5
    want = _device_step(ra, q, k, v, do, P, causal, scale, o_dtype, g_dtype, **kw)
    hin = [_host_tensor(t, pin, pad) for t in (q, k, v, do)]
    hout = _host_outputs(B, N, Hq, Hkv, d, o_dtype, g_dtype, pin, pad)
    _run_host(ra, hin, hout, P, causal, scale, **kw)
    for name, got, ref in zip(("O", "LSE", "dQ", "dK", "dV"), hout, want):
        _same(name, got.contiguous(), ref)
    return q, k, v, do, hout


def _same(name, got, ref):
    """Bit for bit, except dQ: the tensor-core path sums it with reduce-adds
    from many CTAs in an order that varies between runs, so two runs agree to
    fp32 rounding of those sums (relative 1e-5 of the largest entry)."""
    if name.startswith("dQ") and got.dtype == torch.float32:
        tol = 1e-5 * float(ref.abs().max()) + 1e-12
        assert float((got - ref).abs().max()) <= tol, name
    else:
        assert torch.equal(got, ref), name


def test_host_step_bf16_gqa_pinned(ra):
    _case(ra, 2, 1024, 4, 2, 128, 4, True, torch.bfloat16, torch.bfloat16, torch.float32, 81)


def test_host_step_bf16_pageable_and_batch_strided(ra):
    _case(ra, 2, 1024, 2, 2, 128, 4, True, torch.bfloat16, torch.float32, torch.bfloat16, 82, pin=False, pad=128)


def test_host_step_flags_pass_through(ra):
    _case(ra, 1, 2048, 2, 2, 64, 4, True, torch.bfloat16, torch.float32, torch.float32, 83,
          precise=True, striped=True)


def test_host_step_fp32_against_oracle(ra):
    q, k, v, do, hout = _case(ra, 1, 512, 2, 2, 64, 4, False, torch.float32, torch.float32, torch.float32, 84)
    rq, rk, rv, rO, rL, _ = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), False, 64 ** -0.5)
    for name, got, want, kind in (("O", hout[0], rO, "out"), ("LSE", hout[1], rL, "lse"),
                                  ("dQ", hout[2], rq, "out"), ("dK", hout[3], rk, "out"),
                                  ("dV", hout[4], rv, "out")):
        check(f"host step {name}", f64(got), want, torch.float32, kind)


def test_host_step_two_streams_alternating(ra):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    B, N, Hq, Hkv, d, P = 1, 1024, 4, 2, 128, 4
    scale = d ** -0.5
    cases = [make_tensors(B, N, Hq, Hkv, d, torch.bfloat16, "cuda", 90 + i) for i in range(4)]
    wants = [_device_step(ra, *c, P, True, scale, torch.bfloat16, torch.bfloat16) for c in cases]
    hins = [[_host_tensor(t, True) for t in c] for c in cases]
    houts = [_host_outputs(B, N, Hq, Hkv, d, torch.bfloat16, torch.bfloat16, True) for _ in cases]
    sh = ra.shape_of(hins[0][0], hins[0][1])
    nbytes = ra.ra_ring_step_host_workspace_bytes(ra.RA_BF16, ra.RA_BF16, ra.RA_BF16, sh, P)
    wss = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    sts = [torch.cuda.Stream(), torch.cuda.Stream()]
    for i in range(4):   # enqueue all four before waiting on any
        ra.ra_ring_step_host(*hins[i], P, True, scale, *houts[i], wss[i % 2], sts[i % 2])
    for st in sts:
        st.synchronize()
    ra.ra_sync_status(None)
    for i in range(4):
        for name, got, ref in zip(("O", "LSE", "dQ", "dK", "dV"), houts[i], wants[i]):
            _same(f"{name} of call {i}", got, ref)


def test_host_step_rejects_device_tensors(ra):
    t = torch.zeros(1, 256, 1, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RAError):
        ra.ra_ring_step_host(t, t, t, t, 1, True, 0.125, t, t, t, t, t, t)
