"""Pins for the fp64 oracle, independent of the oracle's own formulas.

Each test fixes a value that the mathematics or the pages determine (closed
forms, invariants, brute-force finite differences, a library routine on tiny
inputs), so that a dropped term, a wrong sign or index or a transposed
operand in the oracle fails at least one of them.  The planted-mistake tests
at the end check that claim for the likeliest mistakes.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from oracle import attention as A

RNG = np.random.default_rng(20231001)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# --- closed forms -----------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_visible_values(causal):
    B, N, H, d = 2, 9, 3, 5
    q = rand(B, N, H, d)
    kbar = rand(d)
    k = np.broadcast_to(kbar, (B, N, H, d)).copy()
    v = rand(B, N, H, d)
    scale = 0.37
    O, LSE = oracle.attention_fwd(q, k, v, causal, scale)
    for b, h, i in itertools.product(range(B), range(H), range(N)):
        cnt = i + 1 if causal else N
        np.testing.assert_allclose(O[b, i, h], v[b, :cnt, h].mean(axis=0), atol=1e-13)
        want = scale * (q[b, i, h] @ kbar) + math.log(cnt)
        assert abs(LSE[b, h, i] - want) < 1e-12


def test_single_key_returns_its_value_row():
    B, H, d = 1, 2, 7
    q = rand(B, 4, H, d)
    k = rand(B, 1, H, d)
    v = rand(B, 1, H, d)
    O, LSE = oracle.attention_fwd(q, k, v, False, 0.5)
    for h, i in itertools.product(range(H), range(4)):
        np.testing.assert_array_equal(O[0, i, h], v[0, 0, h])
        assert abs(LSE[0, h, i] - 0.5 * (q[0, i, h] @ k[0, 0, h])) < 1e-13


def test_causal_row_zero_sees_only_key_zero():
    q, k, v = rand(1, 6, 1, 4), rand(1, 6, 1, 4), rand(1, 6, 1, 4)
    O, LSE = oracle.attention_fwd(q, k, v, True, 0.25)
    np.testing.assert_array_equal(O[0, 0, 0], v[0, 0, 0])
    assert abs(LSE[0, 0, 0] - 0.25 * (q[0, 0, 0] @ k[0, 0, 0])) < 1e-14


def test_two_keys_give_sigmoid_weights():
    d = 6
    q, k, v = rand(1, 1, 1, d), rand(1, 2, 1, d), rand(1, 2, 1, d)
    scale = 0.8
    s0 = scale * q[0, 0, 0] @ k[0, 0, 0]
    s1 = scale * q[0, 0, 0] @ k[0, 1, 0]
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    O, LSE = oracle.attention_fwd(q, k, v, False, scale)
    np.testing.assert_allclose(O[0, 0, 0], w0 * v[0, 0, 0] + (1 - w0) * v[0, 1, 0], atol=1e-14)
    assert abs(LSE[0, 0, 0] - np.logaddexp(s0, s1)) < 1e-13


def test_scale_is_inverse_sqrt_head_dim_in_the_pages_example():
    # head_dim ** -0.5 for head_dim 128 is 1/sqrt(128)
    assert 128 ** -0.5 == pytest.approx(1.0 / math.sqrt(128), rel=1e-15)


# --- invariants ---------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one_and_mask_is_lower_triangular(causal):
    q, k = rand(2, 11, 4, 8), rand(2, 11, 2, 8)
    P = oracle.attention_probs(q, k, causal, 0.3)
    assert (P >= 0).all()
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, atol=1e-14)
    if causal:
        assert np.abs(np.triu(P, 1)).max() == 0.0
        assert (np.diagonal(P, axis1=2, axis2=3) > 0).all()


def test_noncausal_output_invariant_to_kv_permutation():
    q, k, v = rand(1, 7, 2, 5), rand(1, 13, 2, 5), rand(1, 13, 2, 5)
    perm = RNG.permutation(13)
    O1, L1 = oracle.attention_fwd(q, k, v, False, 0.6)
    O2, L2 = oracle.attention_fwd(q, k[:, perm], v[:, perm], False, 0.6)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_shifting_every_key_shifts_lse_only(causal):
    q, k, v = rand(1, 8, 2, 4), rand(1, 8, 2, 4), rand(1, 8, 2, 4)
    c = rand(4)
    scale = 0.45
    O1, L1 = oracle.attention_fwd(q, k, v, causal, scale)
    O2, L2 = oracle.attention_fwd(q, k + c, v, causal, scale)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    shift = scale * np.einsum("bnhd,d->bhn", q, c)
    np.testing.assert_allclose(L2 - L1, shift, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 6, 12])
def test_blocked_ring_equals_plain_definition(causal, P):
    q, k, v = rand(2, 12, 4, 6, scale=3.0), rand(2, 12, 2, 6), rand(2, 12, 2, 6)
    O1, L1 = oracle.attention_fwd(q, k, v, causal, 0.7)
    O2, L2 = oracle.ring_fwd_blocked(q, k, v, P, causal, 0.7)
    np.testing.assert_allclose(O2, O1, atol=1e-12, rtol=0)
    np.testing.assert_allclose(L2, L1, atol=1e-12, rtol=0)


def test_ring_schedule_matches_the_pages_rotation():
    # host i computes against its own chunk first, then i-1, i-2, ... (mod P)
    assert oracle.ring_schedule(4, False) == [[0, 3, 2, 1], [1, 0, 3, 2], [2, 1, 0, 3], [3, 2, 1, 0]]
    assert oracle.ring_schedule(4, True) == [[0], [1, 0], [2, 1, 0], [3, 2, 1, 0]]
    for P in (1, 2, 5, 8):
        for blocks in oracle.ring_schedule(P, False):
            assert sorted(blocks) == list(range(P))


def test_merge_identity_commutativity_associativity():
    B, N, H, d = 1, 5, 2, 3
    def tri():
        m = rand(B, H, N)
        return m, np.exp(rand(B, H, N)), rand(B, N, H, d)
    a, b, c = tri(), tri(), tri()
    empty = (np.full((B, H, N), -np.inf), np.zeros((B, H, N)), np.zeros((B, N, H, d)))
    for x, y in zip(oracle.merge_states(empty, a), a):
        np.testing.assert_array_equal(x, y)
    ab = oracle.finalize_state(oracle.merge_states(a, b))
    ba = oracle.finalize_state(oracle.merge_states(b, a))
    np.testing.assert_allclose(ab[0], ba[0], atol=1e-14)
    l1 = oracle.finalize_state(oracle.merge_states(oracle.merge_states(a, b), c))
    l2 = oracle.finalize_state(oracle.merge_states(a, oracle.merge_states(b, c)))
    np.testing.assert_allclose(l1[0], l2[0], atol=1e-13)
    np.testing.assert_allclose(l1[1], l2[1], atol=1e-13)


def test_fully_masked_block_contributes_nothing():
    q, k, v = rand(1, 4, 1, 3), rand(1, 4, 1, 3), rand(1, 4, 1, 3)
    m, l, o = oracle.block_state(q, k, v, True, 1.0, 0, 100)   # every key after every query
    assert np.isneginf(m).all() and (l == 0).all() and (o == 0).all()
    O, LSE = oracle.finalize_state((m, l, o))
    assert (O == 0).all() and np.isneginf(LSE).all()


def test_block_state_with_offsets_matches_full_rows():
    # a Q block at rows 8..11 against a KV block at rows 4..11 (causal)
    q, k, v = rand(1, 12, 2, 4), rand(1, 12, 2, 4), rand(1, 12, 2, 4)
    st = oracle.block_state(q[:, 8:], k[:, 4:], v[:, 4:], True, 0.5, 8, 4)
    st0 = oracle.block_state(q[:, 8:], k[:, :4], v[:, :4], True, 0.5, 8, 0)
    O, L = oracle.finalize_state(oracle.merge_states(st, st0))
    Of, Lf = oracle.attention_fwd(q, k, v, True, 0.5)
    np.testing.assert_allclose(O, Of[:, 8:], atol=1e-13)
    np.testing.assert_allclose(L, Lf[:, :, 8:], atol=1e-13)


# --- gradients ----------------------------------------------------------------

def _loss(q, k, v, do, causal, scale):
    O, _ = oracle.attention_fwd(q, k, v, causal, scale)
    return float((O * do).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_finite_differences(causal):
    B, N, hq, hkv, d = 1, 6, 2, 1, 3
    q, k, v, do = rand(B, N, hq, d), rand(B, N, hkv, d), rand(B, N, hkv, d), rand(B, N, hq, d)
    scale = 0.9
    dq, dk, dv, *_ = oracle.attention_bwd(q, k, v, do, causal, scale)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], do, causal, scale)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], do, causal, scale)
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sum_identities(causal):
    # sum_j dS_ij = 0  =>  sum_j dK_j = 0 ; rows of P sum to 1 => sum_j dV_j = sum_i dO_i
    q, k, v, do = rand(2, 16, 4, 5), rand(2, 16, 2, 5), rand(2, 16, 2, 5), rand(2, 16, 4, 5)
    dq, dk, dv, *_ = oracle.attention_bwd(q, k, v, do, causal, 0.4)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    dosum = do.reshape(2, 16, 2, 2, 5).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), dosum, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_sdpa_fp64(causal):
    torch = pytest.importorskip("torch")
    B, N, hq, hkv, d = 2, 10, 4, 2, 6
    q, k, v, do = rand(B, N, hq, d), rand(B, N, hkv, d), rand(B, N, hkv, d), rand(B, N, hq, d)
    scale = d ** -0.5
    tq = torch.tensor(q).permute(0, 2, 1, 3).requires_grad_()
    tk = torch.tensor(k).permute(0, 2, 1, 3).requires_grad_()
    tv = torch.tensor(v).permute(0, 2, 1, 3).requires_grad_()
    rep = hq // hkv
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(rep, dim=1), tv.repeat_interleave(rep, dim=1),
        is_causal=causal, scale=scale)
    out.backward(torch.tensor(do).permute(0, 2, 1, 3))
    O, _ = oracle.attention_fwd(q, k, v, causal, scale)
    dq, dk, dv, *_ = oracle.attention_bwd(q, k, v, do, causal, scale)
    np.testing.assert_allclose(O, out.detach().permute(0, 2, 1, 3).numpy(), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.permute(0, 2, 1, 3).numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.permute(0, 2, 1, 3).numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.permute(0, 2, 1, 3).numpy(), atol=1e-12)


# --- the row-subsample mode against brute force --------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_row_mode_matches_full(causal):
    B, N, hq, hkv, d = 1, 40, 4, 2, 5
    q, k, v, do = rand(B, N, hq, d), rand(B, N, hkv, d), rand(B, N, hkv, d), rand(B, N, hq, d)
    dq, dk, dv, O, LSE, D = oracle.attention_bwd(q, k, v, do, causal, 0.5)
    rows = [(0, h, i) for h in range(hq) for i in (0, 7, 39)]
    r = oracle.attention_rows(q, k, v, rows, causal, 0.5, do=do)
    for idx, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(r["O"][idx], O[b, i, h], atol=1e-13)
        assert abs(r["LSE"][idx] - LSE[b, h, i]) < 1e-13
        assert abs(r["D"][idx] - D[b, h, i]) < 1e-13
        np.testing.assert_allclose(r["dQ"][idx], dq[b, i, h], atol=1e-13)


def test_last_rows_give_complete_kv_grads_of_last_keys():
    B, N, hq, hkv, d, R = 1, 48, 4, 2, 5, 8
    q, k, v, do = rand(B, N, hq, d), rand(B, N, hkv, d), rand(B, N, hkv, d), rand(B, N, hq, d)
    dq, dk, dv, *_ = oracle.attention_bwd(q, k, v, do, True, 0.5)
    g = 1
    rows = [(0, h, i) for h in (2, 3) for i in range(N - R, N)]
    r = oracle.attention_rows(q, k, v, rows, True, 0.5, do=do, want_kv_grads=True)
    dk_t, dv_t = r["kv_grads"][(0, g)]
    np.testing.assert_allclose(dk_t[N - R:], dk[0, N - R:, g], atol=1e-13)
    np.testing.assert_allclose(dv_t[N - R:], dv[0, N - R:, g], atol=1e-13)


# --- planted mistakes: each must be caught by a pin above ---------------------

def _sketch_merge(a, b):
    """The printed sketch's merge: adds exp_sum-weighted chunk outputs without
    rescaling to a common max (the mistake the pages' own text reports)."""
    ma, la, oa = a
    mb, lb, ob = b
    m = np.maximum(ma, mb)
    return m, la + lb, oa + ob


def test_planted_sketch_merge_is_caught(monkeypatch):
    monkeypatch.setattr(A, "merge_states", _sketch_merge)
    q, k, v = rand(1, 12, 2, 6, scale=3.0), rand(1, 12, 2, 6), rand(1, 12, 2, 6)
    O1, _ = A.attention_fwd(q, k, v, False, 0.7)
    O2, _ = A.ring_fwd_blocked(q, k, v, 4, False, 0.7)
    assert np.abs(O1 - O2).max() > 1e-3


def test_planted_strict_causal_mask_is_caught(monkeypatch):
    def strict(nq, nk, causal, q_off, kv_off):
        qpos = q_off + np.arange(nq)[:, None]
        kpos = kv_off + np.arange(nk)[None, :]
        return (kpos < qpos) if causal else np.ones((nq, nk), bool)
    monkeypatch.setattr(A, "_visible", strict)
    q, k, v = rand(1, 6, 1, 4), rand(1, 6, 1, 4), rand(1, 6, 1, 4)
    O, _ = A.attention_fwd(q, k, v, True, 0.25)
    assert not np.allclose(O[0, 0, 0], v[0, 0, 0])


def test_planted_transposed_kv_head_map_is_caught(monkeypatch):
    monkeypatch.setattr(A, "_kv_head", lambda h, hq, hkv: h % hkv)
    B, N, hq, hkv, d = 1, 5, 4, 2, 3
    q, k, v = rand(B, N, hq, d), rand(B, N, hkv, d), rand(B, N, hkv, d)
    torch = pytest.importorskip("torch")
    O, _ = A.attention_fwd(q, k, v, False, 0.5)
    tq = torch.tensor(q).permute(0, 2, 1, 3)
    tk = torch.tensor(k).permute(0, 2, 1, 3).repeat_interleave(2, dim=1)
    tv = torch.tensor(v).permute(0, 2, 1, 3).repeat_interleave(2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.5)
    assert np.abs(O - ref.permute(0, 2, 1, 3).numpy()).max() > 1e-3


def test_planted_missing_D_term_in_backward_is_caught():
    # dK built from dS = P * dP (the D_i term dropped) breaks sum_j dK_j = 0,
    # which the correct oracle satisfies (test_gradient_sum_identities)
    q, k, v, do = rand(1, 8, 1, 3), rand(1, 8, 1, 3), rand(1, 8, 1, 3), rand(1, 8, 1, 3)
    scale = 0.5
    P = A.attention_probs(q, k, True, scale)[0, 0]
    dP = do[0, :, 0] @ v[0, :, 0].T
    dk_broken = scale * (P * dP).T @ q[0, :, 0]
    assert np.abs(dk_broken.sum(axis=0)).max() > 1e-6
    _, dk, *_ = A.attention_bwd(q, k, v, do, True, scale)
    assert np.abs(dk.sum(axis=1)).max() < 1e-12


# --- striped (load-balanced) ordering -----------------------------------------

def test_striped_positions_are_a_round_robin_permutation():
    pos = oracle.striped_positions(12, 3)
    assert sorted(pos) == list(range(12))
    # host 0 holds 0, 3, 6, 9; host 1 holds 1, 4, 7, 10; host 2 holds 2, 5, 8, 11
    assert list(pos) == [0, 3, 6, 9, 1, 4, 7, 10, 2, 5, 8, 11]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 6])
def test_striped_ring_equals_plain_definition(P):
    N = 12
    q, k, v = rand(2, N, 4, 5, scale=2.0), rand(2, N, 2, 5), rand(2, N, 2, 5)
    pos = oracle.striped_positions(N, P)
    # striped layout: row r holds sequence position pos[r]
    Os, Ls = oracle.ring_fwd_blocked_striped(q[:, pos], k[:, pos], v[:, pos], P, 0.6)
    O, L = oracle.attention_fwd(q, k, v, True, 0.6)
    np.testing.assert_allclose(Os, O[:, pos], atol=1e-12)
    np.testing.assert_allclose(Ls, L[:, :, pos], atol=1e-12)


def test_striped_blocks_share_the_causal_work_evenly():
    # every (query host, key host) pair sees about half of its S x S pairs
    N, P = 64, 4
    S = N // P
    pos = oracle.striped_positions(N, P)
    vis = pos[None, :] <= pos[:, None]
    counts = [[int(vis[i * S:(i + 1) * S, j * S:(j + 1) * S].sum()) for j in range(P)] for i in range(P)]
    for i in range(P):
        for j in range(P):
            assert counts[i][j] == (S * (S + 1) // 2 if j <= i else S * (S - 1) // 2)


# --- variable per-host lengths (dynamic masking) ---------------------------------

def test_varlen_rows_concatenate_valid_prefixes():
    rows = oracle.varlen_rows(12, 3, [2, 4, 0])
    assert list(rows) == [0, 1, 4, 5, 6, 7]


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_with_full_hosts_is_plain_attention(causal):
    q, k, v, do = rand(1, 12, 2, 4), rand(1, 12, 2, 4), rand(1, 12, 2, 4), rand(1, 12, 2, 4)
    a = oracle.attention_varlen(q, k, v, do, 3, [4, 4, 4], causal, 0.5)
    b = oracle.attention_bwd(q, k, v, do, causal, 0.5)
    for x, y in zip(a, b[:5]):
        np.testing.assert_allclose(x, y, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_ignores_padding_values_and_zeroes_padded_rows(causal):
    P, S = 3, 5
    lens = [3, 5, 1]
    q, k, v, do = rand(1, P * S, 2, 4), rand(1, P * S, 1, 4), rand(1, P * S, 1, 4), rand(1, P * S, 2, 4)
    rows = oracle.varlen_rows(P * S, P, lens)
    pad = np.setdiff1d(np.arange(P * S), rows)
    dq, dk, dv, O, L = oracle.attention_varlen(q, k, v, do, P, lens, causal, 0.7)
    # padded rows: nothing computed, nothing leaks out
    assert (O[:, pad] == 0).all() and np.isneginf(L[:, :, pad]).all()
    assert (dq[:, pad] == 0).all() and (dk[:, pad] == 0).all() and (dv[:, pad] == 0).all()
    # changing what sits in the padding changes nothing
    q2, k2, v2, do2 = q.copy(), k.copy(), v.copy(), do.copy()
    for t in (q2, k2, v2, do2):
        t[:, pad] = 1e3 * rand(*t[:, pad].shape)
    res2 = oracle.attention_varlen(q2, k2, v2, do2, P, lens, causal, 0.7)
    for x, y in zip((dq, dk, dv, O, L), res2):
        np.testing.assert_allclose(x, y, atol=1e-12)
    # the valid rows are exactly attention over the packed sequence (brute force)
    Op, Lp = oracle.attention_fwd(q[:, rows], k[:, rows], v[:, rows], causal, 0.7)
    np.testing.assert_allclose(O[:, rows], Op, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_empty_host_drops_out(causal):
    # host 1 holds no tokens: the result is attention over hosts 0 and 2 alone,
    # forward and backward, and host 1's rows are all padding
    P, S = 3, 4
    q, k, v, do = rand(1, P * S, 2, 3), rand(1, P * S, 2, 3), rand(1, P * S, 2, 3), rand(1, P * S, 2, 3)
    dq, dk, dv, O, L = oracle.attention_varlen(q, k, v, do, P, [S, 0, S], causal, 0.9)
    keep = np.r_[0:S, 2 * S:3 * S]
    gq, gk, gv, Ok, Lk, _ = oracle.attention_bwd(q[:, keep], k[:, keep], v[:, keep], do[:, keep], causal, 0.9)
    np.testing.assert_allclose(O[:, keep], Ok, atol=1e-13)
    np.testing.assert_allclose(L[:, :, keep], Lk, atol=1e-13)
    for g, ref in ((dq, gq), (dk, gk), (dv, gv)):
        np.testing.assert_allclose(g[:, keep], ref, atol=1e-13)
        assert (g[:, S:2 * S] == 0).all()
    assert np.isneginf(L[:, :, S:2 * S]).all()


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_all_hosts_empty(causal):
    # no host holds a token: every row is padding, forward and backward
    P, S = 3, 4
    q, k, v, do = rand(1, P * S, 2, 3), rand(1, P * S, 2, 3), rand(1, P * S, 2, 3), rand(1, P * S, 2, 3)
    dq, dk, dv, O, L = oracle.attention_varlen(q, k, v, do, P, [0, 0, 0], causal, 0.9)
    assert (O == 0).all() and np.isneginf(L).all()
    assert (dq == 0).all() and (dk == 0).all() and (dv == 0).all()
    O2, L2 = oracle.attention_varlen(q, k, v, None, P, [0, 0, 0], causal, 0.9)
    assert (O2 == 0).all() and np.isneginf(L2).all()


# --- the row-block mode of the backward against the full matrices ---------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("row_block", [1, 7, 64])
def test_row_block_backward_matches_full(causal, row_block):
    B, N, hq, hkv, d = 2, 37, 4, 2, 5
    q, k, v, do = rand(B, N, hq, d), rand(B, N, hkv, d), rand(B, N, hkv, d), rand(B, N, hq, d)
    dq, dk, dv, O, LSE, D = oracle.attention_bwd(q, k, v, do, causal, 0.45)
    r = oracle.attention_bwd_by_row_blocks(q, k, v, do, causal, 0.45, row_block=row_block)
    for name, got, want in (("O", r["O"], O), ("LSE", r["LSE"], LSE), ("D", r["D"], D), ("dQ", r["dQ"], dq),
                            ("dK", r["dK"], dk), ("dV", r["dV"], dv)):
        np.testing.assert_allclose(got, want, atol=1e-12, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_row_block_backward_selected_keys_and_heads(causal):
    B, N, hq, hkv, d = 1, 50, 4, 2, 6
    q, k, v, do = rand(B, N, hq, d), rand(B, N, hkv, d), rand(B, N, hkv, d), rand(B, N, hq, d)
    keys = np.array([0, 3, 17, 31, 32, 49])
    dq, dk, dv, *_ = oracle.attention_bwd(q, k, v, do, causal, 0.6)
    r = oracle.attention_bwd_by_row_blocks(q, k, v, do, causal, 0.6, keys=keys, want_dq=False, row_block=16)
    np.testing.assert_allclose(r["dK"], dk[:, keys], atol=1e-12)
    np.testing.assert_allclose(r["dV"], dv[:, keys], atol=1e-12)
    assert "dQ" not in r
    # the heads of key/value head 1 only: its dK, dV are complete, head 0's are zero
    r1 = oracle.attention_bwd_by_row_blocks(q, k, v, do, causal, 0.6, keys=keys, heads=[2, 3], row_block=9)
    np.testing.assert_allclose(r1["dK"][:, :, 1], dk[:, keys, 1], atol=1e-12)
    np.testing.assert_allclose(r1["dV"][:, :, 1], dv[:, keys, 1], atol=1e-12)
    assert not r1["dK"][:, :, 0].any() and not r1["dV"][:, :, 0].any()


def test_row_block_backward_key_gradient_by_finite_differences():
    # dK and dV of one selected key against central differences of L = sum(O * dO)
    B, N, hq, hkv, d = 1, 9, 2, 1, 3
    q, k, v, do = rand(B, N, hq, d), rand(B, N, hkv, d), rand(B, N, hkv, d), rand(B, N, hq, d)
    j, eps = 4, 1e-6
    r = oracle.attention_bwd_by_row_blocks(q, k, v, do, True, 0.7, keys=[j], want_dq=False, row_block=2)
    for name, x, g in (("k", k, r["dK"]), ("v", v, r["dV"])):
        for c in range(d):
            xp, xm = x.copy(), x.copy()
            xp[0, j, 0, c] += eps
            xm[0, j, 0, c] -= eps
            kp, vp = (xp, v) if name == "k" else (k, xp)
            km, vm = (xm, v) if name == "k" else (k, xm)
            num = (_loss(q, kp, vp, do, True, 0.7) - _loss(q, km, vm, do, True, 0.7)) / (2 * eps)
            assert abs(g[0, 0, 0, c] - num) < 1e-7 * max(1.0, abs(num)), (name, c)
