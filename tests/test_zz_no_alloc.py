"""The allocation-free ring forward, ra_ring_fwd_noalloc.

Some callers cannot allocate device memory at the point where they run
attention (code inside a host callback or an allocator hook, a framework that
owns every device allocation, a process with a fixed memory budget), so they
cannot hand ra_ring_fwd its workspace.  ra_ring_fwd_noalloc uses a scratch
buffer built into the library instead.  These tests call it through the C ABI
and check it against ra_ring_fwd with a caller workspace -- the two run the
same kernels in the same order, so their outputs must be identical -- and
against the fp64 oracle, on two calls in a row with different inputs (the
shared buffer keeps the first call's data, so the second call must not
depend on it).  They also check that a call takes no device memory, and the
size limit: a shape whose scratch is exactly 32 MiB is accepted, one row more
is refused.  This file sorts last so that a run stopping at the first failure
has run every other test before it.
"""
import ctypes
import os

import pytest
import torch

os.environ.setdefault("RA_WAIT_TIMEOUT_MS", "3000")

import oracle  # noqa: E402
from tests._parity import check, f64  # noqa: E402

pytestmark = pytest.mark.gpu

LIMIT = 32 << 20  # bytes of built-in scratch


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


def _outputs(q):
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(1, q.shape[2], q.shape[1], dtype=torch.float32, device="cuda")
    return o, lse


@pytest.mark.parametrize("causal", [True, False])
def test_noalloc_matches_workspace_entry_point_twice(ra, causal):
    P, scale = 4, 128 ** -0.5
    flags = ra.RA_CAUSAL if causal else 0
    for call, seed in enumerate((501, 502)):
        q, k, v = _inputs(seed)
        o, lse = _outputs(q)
        assert _call_noalloc(ra, q, k, v, P, flags, scale, o, lse) == 0, ra.ra_last_error()
        ra.ra_sync_status()
        o_ref, lse_ref = ra.ring_attention_fwd(q, k, v, P, causal, scale)
        ra.ra_sync_status()
        assert torch.equal(o, o_ref), f"O differs from ra_ring_fwd (call {call + 1})"
        assert torch.equal(lse, lse_ref), f"LSE differs from ra_ring_fwd (call {call + 1})"
        rO, rL = oracle.attention_fwd(f64(q), f64(k), f64(v), causal, scale)
        check(f"noalloc O vs oracle (call {call + 1})", f64(o), rO, torch.bfloat16)
        check(f"noalloc LSE vs oracle (call {call + 1})", f64(lse), rL, torch.bfloat16, kind="lse")


def test_noalloc_takes_no_device_memory(ra):
    q, k, v = _inputs(503)
    o, lse = _outputs(q)
    scale = 128 ** -0.5
    assert _call_noalloc(ra, q, k, v, 4, ra.RA_CAUSAL, scale, o, lse) == 0, ra.ra_last_error()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert _call_noalloc(ra, q, k, v, 4, ra.RA_CAUSAL, scale, o, lse) == 0, ra.ra_last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


def test_noalloc_accepts_exactly_its_scratch_size(ra):
    # fp16 copy of V: 1 * 131072 * 1 * 128 * 2 bytes = 32 MiB exactly, plus
    # the 256-byte unit counter
    N, scale = 131072, 128 ** -0.5
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    q, k, v, _ = make_tensors(1, N, 1, 1, 128, torch.bfloat16, "cuda", 504, with_do=False)
    assert ra.ra_ring_fwd_workspace_bytes(ra.RA_BF16, ra.shape_of(q, k), 32) == LIMIT + 256
    o, lse = _outputs(q)
    assert _call_noalloc(ra, q, k, v, 32, ra.RA_CAUSAL, scale, o, lse) == 0, ra.ra_last_error()
    ra.ra_sync_status()
    o_ref, lse_ref = ra.ring_attention_fwd(q, k, v, 32, True, scale)
    ra.ra_sync_status()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    # the oracle on sampled rows, including the last one (it reads all of V)
    rows = [(0, 0, i) for i in (0, 1, 4095, 4096, 65535, 65536, 100000, N - 1)]
    r = oracle.attention_rows(f64(q), f64(k), f64(v), rows, True, scale)
    idx = torch.tensor([i for _, _, i in rows], device="cuda")
    check("noalloc O rows at the limit", f64(o[0, idx, 0]), r["O"], torch.bfloat16)
    check("noalloc LSE rows at the limit", f64(lse[0, 0, idx]), r["LSE"], torch.bfloat16, kind="lse")


def test_noalloc_rejects_one_row_more(ra):
    # 131073 rows: 131073 * 256 bytes > 32 MiB
    N = 131073
    q = torch.empty(1, N, 1, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = _outputs(q)
    rc = _call_noalloc(ra, q, q, q, 1, ra.RA_CAUSAL, 0.1, o, lse)
    assert rc == 1
    assert "scratch" in ra.ra_last_error()


def test_noalloc_rejects_shapes_far_beyond_its_scratch(ra):
    # fp16 copy of V would need 1 * 65536 * 4 * 128 * 2 = 64 MiB > 32 MiB
    q = torch.empty(1, 65536, 4, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = _outputs(q)
    rc = _call_noalloc(ra, q, q, q, 32, ra.RA_CAUSAL, 0.1, o, lse)
    assert rc == 1
    assert "scratch" in ra.ra_last_error()
