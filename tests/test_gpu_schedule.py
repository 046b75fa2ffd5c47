"""The ring schedule the tensor-core kernels actually run, read back from the
debug visit log (ra_debug_visit_log).

"Ring Attention: Partition Sequence Length, Not Batch" sets the order: at
step s host i holds key/value block (i - s) mod P, so the forward of host i
meets blocks i, i-1, ..., and the gradients of block j travel on to hosts
j, j+1, ... (its "Gotchas and Failure Modes": gradients flow backwards
through the ring).  Under a causal mask a block wholly after a host's
queries is skipped, leaving P (P + 1) / 2 (host, block) pairs per head.
These tests check, per work unit, the exact sequence of tiles loaded, and per
head the set of (query host, key/value block) pairs visited and skipped, for
the contiguous, striped and variable-length layouts.
"""
import os
from collections import defaultdict

import pytest
import torch

os.environ.setdefault("RA_WAIT_TIMEOUT_MS", "3000")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import blockwise_exact_attention_ra_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _logged(ra, fn, capacity=1 << 20):
    """Run fn() with the visit log on; return the records in log order."""
    entries = torch.zeros(capacity, 4, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    ra.ra_debug_visit_log(entries, count)
    try:
        fn()
        ra.ra_sync_status()
    finally:
        ra.ra_debug_visit_log(None, None)
    n = int(count.item())
    assert n <= capacity
    return [tuple(int(x) for x in r) for r in entries[:n].cpu()]


def _inputs(N, Hq, Hkv, seed=4000):
    from blockwise_exact_attention_ra_gb300.inputs import make_tensors
    return make_tensors(1, N, Hq, Hkv, 128, torch.bfloat16, "cuda", seed)


def _units(records, kind):
    """Records of one kernel grouped per unit, in visit order."""
    u = defaultdict(list)
    for k, head, qt, kt in records:
        if k != kind:
            continue
        u[(head, qt) if kind == 0 else (head, kt)].append(kt if kind == 0 else qt)
    return u


def _dedupe(seq):
    out = []
    for x in seq:
        if not out or out[-1] != x:
            out.append(x)
    return out


# --- expected schedules (the ring order of the pages, per 128-row tile) -------------

def _fwd_expected(N, P, causal, host_len=None):
    """{first query tile of a unit: key/value tiles in visit order} for one head."""
    T = N // P // 128
    nT = N // 128
    exp = {}
    for host in range(P):
        for lp in range((T + 1) // 2):
            ta = host * T + 2 * lp
            tiles = [ta] + ([ta + 1] if 2 * lp + 1 < T else [])
            if host_len is not None:
                tiles = [t for t in tiles if (t - host * T) * 128 < host_len[host]]
                if not tiles:
                    continue
            lead = tiles[-1]
            if causal:
                seq = list(range(lead, -1, -1))
            else:
                top = (host + 1) * T - 1
                seq = [(top - i) % nT for i in range(nT)]
            if host_len is not None:
                seq = [kt for kt in seq if (kt % T) * 128 < host_len[kt // T]]
            exp[ta] = seq
    return exp


def _bwd_expected(N, P, causal, group, host_len=None):
    """{key/value tile: [(query head within the group, query tile)] in visit order}."""
    T = N // P // 128
    nT = N // 128
    exp = {}
    for jt in range(nT):
        if host_len is not None and (jt % T) * 128 >= host_len[jt // T]:
            continue
        seq = []
        for hh in range(group):
            qts = list(range(jt, nT)) if causal else [((jt // T) * T + k) % nT for k in range(nT)]
            if host_len is not None:
                qts = [qt for qt in qts if (qt % T) * 128 < host_len[qt // T]]
            seq += [(hh, qt) for qt in qts]
        exp[jt] = seq
    return exp


@pytest.mark.parametrize("causal", [True, False])
def test_contiguous_ring_schedule(ra, causal):
    N, Hq, Hkv, P = 4096, 4, 2, 8
    T, group = N // P // 128, Hq // Hkv
    q, k, v, do = _inputs(N, Hq, Hkv)

    def run():
        o, lse = ra.ring_attention_fwd(q, k, v, P, causal)
        ra.ring_attention_bwd(q, k, v, o, lse, do, P, causal)

    rec = _logged(ra, run)
    fwd = _units(rec, 0)
    exp_f = _fwd_expected(N, P, causal)
    assert sorted(fwd) == sorted((h, ta) for h in range(Hq) for ta in exp_f)
    for (h, ta), seq in fwd.items():
        assert seq == exp_f[ta], f"forward unit (head {h}, tile {ta})"
    exp_b = _bwd_expected(N, P, causal, group)
    # the backward records carry the query head; regroup per key/value head
    per_unit = defaultdict(list)
    for kind, head, qt, kt in rec:
        if kind == 1:
            per_unit[(head // group, kt)].append((head % group, qt))
    assert len(per_unit) == Hkv * len(exp_b)
    for (g, jt), seq in per_unit.items():
        assert seq == exp_b[jt], f"backward unit (kv head {g}, tile {jt})"
    # (query host, key/value block) pairs per head: the ring order of blocks and,
    # under the mask, exactly P (P + 1) / 2 of the P^2 pairs
    for h in range(Hq):
        pairs = {(ta // T, kt // T) for (hh, ta), seq in fwd.items() if hh == h for kt in seq}
        assert len(pairs) == (P * (P + 1) // 2 if causal else P * P)
        skipped = {(i, j) for i in range(P) for j in range(P)} - pairs
        assert skipped == ({(i, j) for i in range(P) for j in range(P) if j > i} if causal else set())
        for (hh, ta), seq in fwd.items():
            if hh == h:
                i = ta // T
                blocks = _dedupe([kt // T for kt in seq])
                assert blocks == [(i - s) % P for s in range(P)][:len(blocks)]
        bpairs = {(qt // T, jt // T) for (g, jt), seq in per_unit.items() if g == h // group
                  for hh, qt in seq if hh == h % group}
        assert bpairs == pairs
        for (g, jt), seq in per_unit.items():
            j = jt // T
            hosts = _dedupe([qt // T for hh, qt in seq if hh == 0])
            assert hosts == [(j + s) % P for s in range(P)][:len(hosts)]


def test_striped_ring_schedule(ra):
    N, H, P = 4096, 2, 8
    T = N // P // 128
    q, k, v, do = _inputs(N, H, H)

    def run():
        o, lse = ra.ring_attention_fwd(q, k, v, P, True, striped=True)
        ra.ring_attention_bwd(q, k, v, o, lse, do, P, True, striped=True)

    rec = _logged(ra, run)
    fwd = _units(rec, 0)
    # host i, local tiles (2lp, 2lp+1): every block in ring order, local tiles lead..0
    for (h, ta), seq in fwd.items():
        host, lt = divmod(ta, T)
        lead = lt + 1 if lt + 1 < T else lt
        want = [((host - s) % P) * T + t for s in range(P) for t in range(lead, -1, -1)]
        assert seq == want, f"striped forward unit (head {h}, tile {ta})"
    assert len(fwd) == H * P * ((T + 1) // 2)
    bwd = _units(rec, 1)
    assert len(bwd) == H * P * T
    for (h, jt), seq in bwd.items():
        # key tile tk of host j: one lap of the ring per local query tile it
        # meets (tk, tk+1, ...), each lap over hosts j, j+1, ... in ring order
        host, tk = divmod(jt, T)
        want = [((host + s) % P) * T + t for t in range(tk, T) for s in range(P)]
        assert seq == want, f"striped backward unit (head {h}, tile {jt})"


def test_variable_length_schedule_skips_padding(ra):
    N, H, P = 8192, 2, 8
    S = N // P
    T = S // 128
    lens = [S, 0, 300, 128, 1, S - 1, 700, 129]
    hl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q, k, v, do = _inputs(N, H, H)

    def run():
        o, lse = ra.ring_attention_fwd(q, k, v, P, True, host_len=hl)
        ra.ring_attention_bwd(q, k, v, o, lse, do, P, True, host_len=hl)

    rec = _logged(ra, run)
    fwd = _units(rec, 0)
    exp_f = _fwd_expected(N, P, True, lens)
    assert sorted(fwd) == sorted((h, ta) for h in range(H) for ta in exp_f)
    for (h, ta), seq in fwd.items():
        assert seq == exp_f[ta], f"varlen forward unit (head {h}, tile {ta})"
    exp_b = _bwd_expected(N, P, True, 1, lens)
    bwd = _units(rec, 1)
    assert sorted(bwd) == sorted((h, jt) for h in range(H) for jt in exp_b)
    for (h, jt), seq in bwd.items():
        assert seq == [qt for _, qt in exp_b[jt]], f"varlen backward unit (head {h}, tile {jt})"
    # no record touches a tile wholly in padding; host 1 (empty) never appears
    for kind, head, qt, kt in rec:
        for t in (qt, kt):
            assert (t % T) * 128 < lens[t // T], f"padding tile {t} was loaded"


def test_log_is_off_by_default_and_counts_past_capacity(ra):
    N, H, P = 2048, 1, 4
    q, k, v, _ = _inputs(N, H, H)
    entries = torch.zeros(8, 4, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    ra.ra_debug_visit_log(entries, count)
    ra.ring_attention_fwd(q, k, v, P, True)
    ra.ra_sync_status()
    ra.ra_debug_visit_log(None, None)
    total = sum(len(s) for s in _fwd_expected(N, P, True).values())
    assert int(count.item()) == total > 8
    ra.ring_attention_fwd(q, k, v, P, True)   # logging off: nothing more is counted
    ra.ra_sync_status()
    assert int(count.item()) == total
