"""The allocation-free ring forward, ra_ring_fwd_noalloc.

Some callers cannot allocate device memory at the point where they run
attention (code inside a host callback or an allocator hook, a framework that
owns every device allocation, a process with a fixed memory budget), so they
cannot hand ra_ring_fwd its workspace.  ra_ring_fwd_noalloc uses a scratch
buffer built into the library instead.  These tests call it through the C ABI
and check it against ra_ring_fwd with a caller workspace, on two calls in a
row with different inputs (the shared buffer keeps the first call's data, so
the second call must not depend on it).  This file sorts last so that a run
stopping at the first failure has run every other test before it.
"""
import ctypes
import os

import pytest
import torch

os.environ.setdefault("RA_WAIT_TIMEOUT_MS", "3000")

from tests._parity import check, f64  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import blockwise_exact_attention_ra_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _inputs(seed, N=2048, Hq=4, Hkv=2, d=128):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    return make_tensors(1, N, Hq, Hkv, d, torch.bfloat16, "cuda", seed, with_do=False)[:3]


def _call_noalloc(ra, q, k, v, P, flags, scale, o, lse):
    """Direct C-ABI call (ctypes), no torch-side allocation in between."""
    shape = ra.shape_of(q, k)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ra.lib.ra_ring_fwd_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ra.RA_BF16, shape, P, flags, ctypes.c_float(scale), ctypes.c_void_p(o.data_ptr()), ra.RA_F32,
        ctypes.c_void_p(lse.data_ptr()), stream)


@pytest.mark.parametrize("causal", [True, False])
def test_noalloc_matches_workspace_entry_point_twice(ra, causal):
    P, scale = 4, 128 ** -0.5
    flags = ra.RA_CAUSAL if causal else 0
    for call, seed in enumerate((501, 502)):
        q, k, v = _inputs(seed)
        o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        lse = torch.empty(1, q.shape[2], q.shape[1], dtype=torch.float32, device="cuda")
        assert _call_noalloc(ra, q, k, v, P, flags, scale, o, lse) == 0, ra.ra_last_error()
        ra.ra_sync_status()
        o_ref, lse_ref = ra.ring_attention_fwd(q, k, v, P, causal, scale)
        ra.ra_sync_status()
        check(f"noalloc O (call {call + 1})", f64(o), f64(o_ref), torch.bfloat16)
        check(f"noalloc LSE (call {call + 1})", f64(lse), f64(lse_ref), torch.bfloat16, kind="lse")


def test_noalloc_rejects_shapes_beyond_its_scratch(ra):
    # fp16 copy of V would need 1 * 65536 * 4 * 128 * 2 = 64 MiB > 32 MiB
    q = torch.empty(1, 65536, 4, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(1, 4, 65536, dtype=torch.float32, device="cuda")
    rc = _call_noalloc(ra, q, q, q, 32, ra.RA_CAUSAL, 0.1, o, lse)
    assert rc == 1
    assert "scratch" in ra.ra_last_error()
