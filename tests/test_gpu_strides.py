"""Row, head and batch strides through the C ABI.

The pages lay tensors out as [seq, heads, head_dim] ("Building Ring Attention
in PyTorch: The 200-Line Version"); callers also hold [B, H, N, d] tensors or
slices of a fused q/k/v projection.  These run through the same kernels with
their strides passed in ra_shape: outputs are compared with the fp64 oracle,
and with the same computation on packed copies, which visits the same tiles
in the same order and must give identical O, LSE, dK and dV (dQ differs only
by the order of its fp32 reduce-adds).
"""
import ctypes
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


def _head_major(t):
    """The same values held as a [B, H, N, d] tensor, viewed as [B, N, H, d]."""
    return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


def _inputs(B, N, Hq, Hkv, d, dtype, seed):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    return make_tensors(B, N, Hq, Hkv, d, dtype, "cuda", seed)


def _run(ra, q, k, v, do, P, causal, **kw):
    o, lse = ra.ring_attention_fwd(q, k, v, P, causal, **kw)
    dq, dk, dv = ra.ring_attention_bwd(q, k, v, o, lse, do, P, causal, **kw)
    ra.ra_sync_status()
    return o, lse, dq, dk, dv


def _compare(name, strided, packed, dtype, want=None):
    o, lse, dq, dk, dv = strided
    po, plse, pdq, pdk, pdv = packed
    assert torch.equal(o, po), f"{name}: O differs from the packed run"
    assert torch.equal(lse, plse), f"{name}: LSE differs from the packed run"
    assert torch.equal(dk, pdk), f"{name}: dK differs from the packed run"
    assert torch.equal(dv, pdv), f"{name}: dV differs from the packed run"
    diff = (dq - pdq).abs().max().item()
    assert diff <= 1e-5 * max(1.0, pdq.abs().max().item()), f"{name}: dQ differs by {diff:.3e}"
    if want is not None:
        rq, rk, rv, rO, rL = want
        check(f"{name} O", f64(o), rO, dtype)
        check(f"{name} LSE", f64(lse), rL, dtype, kind="lse")
        check(f"{name} dQ", f64(dq), rq, dtype)
        check(f"{name} dK", f64(dk), rk, dtype)
        check(f"{name} dV", f64(dv), rv, dtype)


@pytest.mark.parametrize("dtype,causal", [(torch.bfloat16, True), (torch.bfloat16, False),
                                          (torch.float16, True), (torch.float32, True)])
def test_head_major_tensors(ra, dtype, causal):
    B, N, Hq, Hkv, P = 2, 1024, 4, 2, 4
    d = 64 if dtype == torch.float32 else 128
    q, k, v, do = _inputs(B, N, Hq, Hkv, d, dtype, 5100 + int(causal))
    hq, hk, hv, hdo = (_head_major(t) for t in (q, k, v, do))
    assert hq.stride(1) == d and hq.stride(2) == N * d   # rows at stride d, heads at N*d
    strided = _run(ra, hq, hk, hv, hdo, P, causal)
    assert strided[0].stride() == hq.stride()             # outputs keep the layout
    packed = _run(ra, q, k, v, do, P, causal)
    rq, rk, rv, rO, rL, _ = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), causal, d ** -0.5)
    _compare(f"[B,H,N,d] {dtype}", strided, packed, dtype, (rq, rk, rv, rO, rL))


def test_fused_qkv_slices(ra):
    B, N, H, d, P = 1, 2048, 2, 128, 8
    q, k, v, do = _inputs(B, N, H, H, d, torch.bfloat16, 5110)
    qkv = torch.stack([q, k, v], dim=2)                   # [B, N, 3, H, d]
    fq, fk, fv = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    assert fq.stride(1) == 3 * H * d
    fdo = ra.empty_like_layout(fq)
    fdo.copy_(do)
    strided = _run(ra, fq, fk, fv, fdo, P, True)
    packed = _run(ra, q, k, v, do, P, True)
    _compare("fused q/k/v slices", strided, packed, torch.bfloat16)


@pytest.mark.parametrize("layout", ["striped", "varlen"])
def test_head_major_striped_and_variable_lengths(ra, layout):
    B, N, H, d, P = 1, 2048, 2, 128, 8
    q, k, v, do = _inputs(B, N, H, H, d, torch.bfloat16, 5120)
    kw = {"striped": True} if layout == "striped" else {
        "host_len": torch.tensor([256, 0, 100, 256, 1, 255, 128, 129], dtype=torch.int32, device="cuda")}
    hq, hk, hv, hdo = (_head_major(t) for t in (q, k, v, do))
    strided = _run(ra, hq, hk, hv, hdo, P, True, **kw)
    packed = _run(ra, q, k, v, do, P, True, **kw)
    _compare(f"[B,H,N,d] {layout}", strided, packed, torch.bfloat16)


def test_block_step_and_finalize_with_strides(ra):
    Nq, Nkv, H, d = 384, 256, 2, 128
    q, k, v, _ = _inputs(1, Nq, H, H, d, torch.bfloat16, 5130)
    k, v = k[:, :Nkv], v[:, :Nkv]
    hq, hk, hv = (_head_major(t) for t in (q, k, v))
    sh = ra.shape_of(hq, hk)
    assert sh.q_hstride == Nq * d and sh.kv_hstride == Nkv * d
    o = torch.empty(1, Nq, H, d, device="cuda")
    m = torch.empty(1, H, Nq, device="cuda")
    l = torch.empty(1, H, Nq, device="cuda")
    ra.ra_acc_init(o, m, l, sh)
    ws = torch.empty(ra.ra_block_fwd_workspace_bytes(ra.RA_BF16, sh), dtype=torch.uint8, device="cuda")
    ra.ra_block_fwd(hq, hk, hv, o, m, l, 200, 0, True, d ** -0.5, ws, shape=sh)
    out = ra.empty_like_layout(hq, torch.float32)
    lse = torch.empty(1, H, Nq, device="cuda")
    ra.ra_finalize(o, m, l, out, lse, sh)
    ra.ra_sync_status()
    rm, rl, ro = oracle.block_state(f64(q), f64(k), f64(v), True, d ** -0.5, 200, 0)
    rO, rL = oracle.finalize_state((rm, rl, ro))
    check("strided block O", f64(out), rO, torch.bfloat16)
    check("strided block LSE", f64(lse), rL, torch.bfloat16, kind="lse")


def test_tensor_core_strides_must_be_16_byte_multiples(ra):
    # row and head strides of 260 and 132 bf16 elements are not 16-byte multiples:
    # refused before anything is launched (the buffers cover every offset the
    # strides reach, 255 * 260 + 132 + 128 elements, regardless)
    buf = torch.zeros(1 << 17, dtype=torch.bfloat16, device="cuda")
    o = torch.empty(1 << 17, device="cuda")
    lse = torch.empty(1, 2, 256, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    sh = ra.RaShape(1, 256, 256, 2, 2, 128, 0, 0, 2 * 128 + 4, 128 + 4, 0, 0)
    vp = ctypes.c_void_p
    rc = ra.lib.ra_ring_fwd(vp(buf.data_ptr()), vp(buf.data_ptr()), vp(buf.data_ptr()), ra.RA_BF16, sh, 2, 1,
                            ctypes.c_float(0.1), vp(o.data_ptr()), ra.RA_F32, vp(lse.data_ptr()),
                            vp(ws.data_ptr()), ws.numel(), None)
    assert rc == 1 and "multiples of 8" in ra.ra_last_error()
