"""Multi-process host logic of bench.py on CPU (gloo, world size 2): the step
time is the maximum over ranks and the value counts the work of every rank
(independent replicas; the path has no data exchange between GPUs)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    dist.barrier()
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")   # rank 1 is the slow one
    out[rank] = (ms, bench.job_value(ws, 2.0e12, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    assert out[0] == out[1]
    ms, value = out[0]
    assert ms == pytest.approx(15.0)
    assert value == pytest.approx(2 * 2.0e12 / 15e-3 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_value(1, 1e12, 1000.0) == pytest.approx(1.0)


# ---------------------------------------------------------------------------
# The ring protocol of a multi-GPU run, on CPU ranks.  "Ring Attention:
# Partition Sequence Length, Not Batch": host i sends the key/value block it
# holds to host i+1 and receives the next one from host i-1, so at step s it
# holds block (i - s) mod P; "The Synchronous Send/Recv Trap": post the
# transfer before computing on the held block and wait for it afterwards.
# The backward sends each block on with its dK, dV accumulators, so they
# visit hosts j, j+1, ... and are back with their owner after P hops.  The
# per-block arithmetic here is the oracle's; what is checked is the order of
# the exchange and that it composes to the whole-sequence result.
# ---------------------------------------------------------------------------

RING_P, RING_S = 4, 16


def _ring_worker(rank, world, port, causal, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    import oracle
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    q, k, v, _ = make_tensors(1, RING_P * RING_S, 2, 2, 8, torch.float64, "cpu", 2024, with_do=False)
    scale = 8 ** -0.5
    S, i = RING_S, rank
    rows = slice(i * S, (i + 1) * S)
    held = torch.cat([k[:, rows], v[:, rows]]).contiguous()   # the block travels as one buffer
    held_id = torch.tensor([i], dtype=torch.int64)
    acc = (np.full((1, 2, S), -np.inf), np.zeros((1, 2, S)), np.zeros((1, S, 2, 8)))
    seen, computed = [], []
    for s in range(world):
        reqs = []
        if s < world - 1:   # post the exchange first, compute on the held block meanwhile
            nxt, nxt_id = torch.empty_like(held), torch.empty_like(held_id)
            reqs = [dist.isend(held, (i + 1) % world), dist.isend(held_id, (i + 1) % world),
                    dist.irecv(nxt, (i - 1) % world), dist.irecv(nxt_id, (i - 1) % world)]
        j = int(held_id)
        seen.append(j)
        if not (causal and j > i):   # blocks wholly in this host's causal future are skipped
            part = oracle.block_state(q[:, rows].numpy(), held[:1].numpy(), held[1:].numpy(), causal, scale,
                                      i * S, j * S)
            acc = oracle.merge_states(acc, part)
            computed.append(j)
        for r in reqs:
            r.wait()
        if reqs:
            held, held_id = nxt, nxt_id
    O, LSE = oracle.finalize_state(acc)
    # backward hops: each block's accumulator records the hosts it visits, in order
    trail = torch.full((world,), -1, dtype=torch.int64)
    trail_owner = torch.tensor([i], dtype=torch.int64)
    for s in range(world):
        trail[s] = i          # host i adds its queries' contribution at hop s
        nxt, nxt_owner = torch.empty_like(trail), torch.empty_like(trail_owner)
        reqs = [dist.isend(trail, (i + 1) % world), dist.isend(trail_owner, (i + 1) % world),
                dist.irecv(nxt, (i - 1) % world), dist.irecv(nxt_owner, (i - 1) % world)]
        for r in reqs:
            r.wait()
        trail, trail_owner = nxt, nxt_owner
    out[rank] = (seen, computed, O, LSE, trail.tolist(), int(trail_owner))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("causal", [True, False])
def test_ring_exchange_order_and_result_with_gloo_ranks(causal):
    import numpy as np
    import oracle
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_ring_worker, args=(RING_P, _free_port(), causal, out), nprocs=RING_P, join=True)
    q, k, v, _ = make_tensors(1, RING_P * RING_S, 2, 2, 8, torch.float64, "cpu", 2024, with_do=False)
    O_ref, L_ref = oracle.attention_fwd(q.numpy(), k.numpy(), v.numpy(), causal, 8 ** -0.5)
    sched = oracle.ring_schedule(RING_P, causal)
    for i in range(RING_P):
        seen, computed, O, LSE, trail, owner = out[i]
        assert seen == [(i - s) % RING_P for s in range(RING_P)]
        assert computed == sched[i]
        rows = slice(i * RING_S, (i + 1) * RING_S)
        assert np.allclose(O, O_ref[:, rows], rtol=0, atol=1e-12)
        assert np.allclose(LSE, L_ref[:, :, rows], rtol=0, atol=1e-12)
        # after P hops host i holds its own block's accumulators again, which
        # visited hosts i, i+1, ..., i+P-1 in that order
        assert owner == i
        assert trail == [(i + s) % RING_P for s in range(RING_P)]
