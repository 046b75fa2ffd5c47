"""The ring forward and backward captured into a CUDA graph and replayed, and
the workspace the forward needs for its work counter.

Every launch of a call goes to the caller's stream and the workspaces are the
caller's, so a training step can be captured once and replayed; that includes
the work counters the kernels' CTAs draw units from, which each call zeroes in
its workspace before the launch.  A replay that kept a counter from the last
run would find every unit taken and write nothing, so the replays are checked
against the eager results (bitwise where the kernels are deterministic: O, LSE,
dK, dV; dQ is summed by reduce-adds in an order that varies).
"""
import os

import pytest
import torch

os.environ.setdefault("RA_WAIT_TIMEOUT_MS", "3000")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import blockwise_exact_attention_ra_gb300 as ra
    assert torch.cuda.is_available()
    return ra


@pytest.mark.parametrize("striped", [False, True])
def test_ring_step_replays_from_a_cuda_graph(ra, striped):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    B, N, H, d, P = 1, 4096, 2, 128, 4
    q, k, v, do = make_tensors(B, N, H, H, d, torch.bfloat16, "cuda", 77)
    scale = d ** -0.5
    sh = ra.shape_of(q, k)
    wsf = torch.empty(max(16, ra.ra_ring_fwd_workspace_bytes(ra.RA_BF16, sh, P)), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(max(16, ra.ra_ring_bwd_workspace_bytes(ra.RA_BF16, ra.RA_F32, sh, P)), dtype=torch.uint8,
                      device="cuda")
    o = torch.empty(B, N, H, d, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty(B, N, H, d, dtype=torch.float32, device="cuda") for _ in range(3))
    stream = torch.cuda.Stream()

    def step():
        ra.ra_ring_fwd(q, k, v, P, True, scale, o, lse, wsf, stream, striped=striped)
        ra.ra_ring_bwd(q, k, v, o, do, lse, P, True, scale, dq, dk, dv, wsb, stream, striped=striped)

    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step()   # eager: also sets up the device status word and kernel attributes
    stream.synchronize()
    ra.ra_sync_status()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(2):
        for t in (o, lse, dq, dk, dv):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ra.ra_sync_status()
        for name, got, want in zip(("O", "LSE", "dK", "dV"), (o, lse, dk, dv), (ref[0], ref[1], ref[3], ref[4])):
            assert torch.equal(got, want), name
        err = (dq - ref[2]).abs().max().item()
        assert err <= 1e-5 * ref[2].abs().max().item(), f"dQ differs by {err}"


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_ring_fwd_refuses_a_workspace_without_room_for_its_counter(ra, dtype):
    # the 16-bit forward draws its work from a counter in the workspace, fp16
    # inputs included: a missing or short workspace is refused before any launch
    import ctypes
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    q, k, v, _ = make_tensors(1, 512, 2, 2, 128, dtype, "cuda", 78, with_do=False)
    sh = ra.shape_of(q, k)
    need = ra.ra_ring_fwd_workspace_bytes(ra._dt(q), sh, 2)
    assert need >= 256
    o = torch.empty(1, 512, 2, 128, device="cuda")
    lse = torch.empty(1, 2, 512, device="cuda")
    vp = ctypes.c_void_p
    args = [vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), ra._dt(q), sh, 2, 1, ctypes.c_float(0.1),
            vp(o.data_ptr()), ra.RA_F32, vp(lse.data_ptr())]
    assert ra.lib.ra_ring_fwd(*args, None, 0, None) == 1
    assert "workspace" in ra.ra_last_error()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert ra.lib.ra_ring_fwd(*args, vp(ws.data_ptr()), need - 1, None) == 1
    assert ra.lib.ra_ring_fwd(*args, vp(ws.data_ptr()), need, None) == 0, ra.ra_last_error()
    ra.ra_sync_status()
