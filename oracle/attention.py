"""Plain fp64 CPU oracle for exact softmax attention, its gradients and the
blockwise ring schedule.

TEST INFRASTRUCTURE ONLY.  Nothing on the CUDA product path imports or calls
this module; it shares no code, header, table or helper with it.  Inputs are
the exact values handed to the GPU, upcast to float64.

Sources (page title, section):

* "Ring Attention: Train 1M Tokens on 8GB GPUs in 2026", section "Why Standard
  Attention Explodes Past 100K Tokens": Attention(Q, K, V) =
  softmax(Q K^T / sqrt(d_k)) V with Q, K, V in R^{N x d}.
* same page, "Building Ring Attention in PyTorch: The 200-Line Version":
  tensors laid out [seq, heads, head_dim]; scale = head_dim ** -0.5; the ring
  loop visits one KV chunk per step; the output is divided by the softmax
  denominator at the end.
* same page, "Ring Attention: Partition Sequence Length, Not Batch": host i
  owns rows [i N/P, (i+1) N/P); at every step each host passes its KV chunk to
  host i+1 and takes host i-1's, P steps in all.
* same page, "Gotchas and Failure Modes": partial results are carried as the
  triple (max_score, exp_sum, weighted_output) and rescaled when merged.  The
  printed sketch adds chunk results without the exp(m_chunk - m_new) factor;
  its own text calls that a bug, so the oracle follows the rescaled triple
  (online normaliser, Milakov & Gimelshein, cited on the arXiv 2310.01889 page
  "Ring Attention with Blockwise Transformers for Near-Infinite Context").
* "Ring Attention with Blockwise Transformers for Near-Infinite Context",
  Abstract: the blockwise result is exact ("without resorting to
  approximations"), so the plain definition is the reference and the blocked
  mode below must agree with it to rounding.

Readings where the pages are silent (each listed in the design notes):
causal masking keeps key position <= query position (global positions,
contiguous host blocks); grouped-query heads map query head h to key/value
head h // (Hq / Hkv); a row that sees no key has m = -inf, l = 0, O = 0 and
LSE = -inf; the backward pass differentiates L = sum(O * dO).

Layout everywhere: [B, N, H, d] (the pages' [seq, heads, head_dim] plus a
batch axis); LSE and the (m, l) state are [B, H, N].
"""
import numpy as np

NEG_INF = -np.inf


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _kv_head(h, hq, hkv):
    """Query head h reads key/value head h // (Hq/Hkv) (grouped heads)."""
    return h // (hq // hkv)


def _visible(nq, nk, causal, q_off, kv_off, q_pos=None, kv_pos=None):
    """Boolean [nq, nk]: key j visible to query i.  Positions are q_off + i
    and kv_off + j, or the explicit arrays q_pos, kv_pos when given."""
    if not causal:
        return np.ones((nq, nk), dtype=bool)
    qpos = (q_off + np.arange(nq) if q_pos is None else np.asarray(q_pos))[:, None]
    kpos = (kv_off + np.arange(nk) if kv_pos is None else np.asarray(kv_pos))[None, :]
    return kpos <= qpos


def _scores(q2, k2, scale, vis):
    """s_ij = scale * q_i . k_j on visible pairs, -inf elsewhere."""
    s = scale * (q2 @ k2.T)
    return np.where(vis, s, NEG_INF)


def _row_lse(s):
    """LSE_i = m_i + log sum_j exp(s_ij - m_i); -inf for an empty row."""
    m = s.max(axis=1)
    out = np.full(s.shape[0], NEG_INF)
    ok = np.isfinite(m)
    if ok.any():
        e = np.exp(s[ok] - m[ok, None])
        out[ok] = m[ok] + np.log(e.sum(axis=1))
    return out


def attention_probs(q, k, causal, scale, q_off=0, kv_off=0):
    """Softmax matrix P [B, Hq, Nq, Nk] (small cases only).

    Row i is exp(s_i - LSE_i); an empty row is all zeros.
    """
    q, k = _f64(q), _f64(k)
    B, nq, hq, _ = q.shape
    nk, hkv = k.shape[1], k.shape[2]
    vis = _visible(nq, nk, causal, q_off, kv_off)
    P = np.zeros((B, hq, nq, nk))
    for b in range(B):
        for h in range(hq):
            s = _scores(q[b, :, h], k[b, :, _kv_head(h, hq, hkv)], scale, vis)
            lse = _row_lse(s)
            ok = np.isfinite(lse)
            P[b, h, ok] = np.exp(s[ok] - lse[ok, None])
    return P


def attention_fwd(q, k, v, causal, scale, q_off=0, kv_off=0):
    """Exact attention: O = softmax(scale Q K^T) V per (batch, head).

    Returns (O [B, Nq, Hq, d], LSE [B, Hq, Nq]) in float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, nq, hq, d = q.shape
    nk, hkv = k.shape[1], k.shape[2]
    vis = _visible(nq, nk, causal, q_off, kv_off)
    O = np.zeros((B, nq, hq, d))
    LSE = np.full((B, hq, nq), NEG_INF)
    for b in range(B):
        for h in range(hq):
            g = _kv_head(h, hq, hkv)
            s = _scores(q[b, :, h], k[b, :, g], scale, vis)
            lse = _row_lse(s)
            ok = np.isfinite(lse)
            P = np.zeros_like(s)
            P[ok] = np.exp(s[ok] - lse[ok, None])
            O[b, :, h] = P @ v[b, :, g]
            LSE[b, h] = lse
    return O, LSE


def attention_bwd(q, k, v, do, causal, scale):
    """Gradients of L = sum(O * dO) for exact attention (self-attention, q_off = kv_off = 0).

    P = exp(S - LSE); dV_j = sum_i P_ij dO_i; dP_ij = dO_i . v_j;
    D_i = dO_i . O_i; dS_ij = P_ij (dP_ij - D_i); dQ_i = scale sum_j dS_ij k_j;
    dK_j = scale sum_i dS_ij q_i.  Grouped heads sum dK, dV over the group.
    Returns (dQ, dK, dV, O, LSE, D) in float64.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, n, hq, d = q.shape
    hkv = k.shape[2]
    vis = _visible(n, k.shape[1], causal, 0, 0)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    O = np.zeros_like(q)
    LSE = np.full((B, hq, n), NEG_INF)
    Dd = np.zeros((B, hq, n))
    for b in range(B):
        for h in range(hq):
            g = _kv_head(h, hq, hkv)
            s = _scores(q[b, :, h], k[b, :, g], scale, vis)
            lse = _row_lse(s)
            ok = np.isfinite(lse)
            P = np.zeros_like(s)
            P[ok] = np.exp(s[ok] - lse[ok, None])
            o = P @ v[b, :, g]
            D = (do[b, :, h] * o).sum(axis=1)
            dP = do[b, :, h] @ v[b, :, g].T
            dS = P * (dP - D[:, None])
            dq[b, :, h] = scale * (dS @ k[b, :, g])
            dk[b, :, g] += scale * (dS.T @ q[b, :, h])
            dv[b, :, g] += P.T @ do[b, :, h]
            O[b, :, h] = o
            LSE[b, h] = lse
            Dd[b, h] = D
    return dq, dk, dv, O, LSE, Dd


def attention_rows(q, k, v, rows, causal, scale, do=None, want_kv_grads=False):
    """Forward (and optionally backward) of selected query rows only.

    ``rows`` is a sequence of (b, h, i).  Each row is computed from the plain
    definition against every key it sees (no blocking).  Returns a dict with
    O [R, d], LSE [R]; with ``do`` given also D [R] and dQ [R, d]; with
    ``want_kv_grads`` also the contributions of exactly these rows to dK and
    dV as dicts {(b, g): (dK [Nk, d], dV [Nk, d])}.  Under a causal mask the
    last R query rows of every head of a group are the only rows that see the
    last R keys, so their contributions are the complete dK, dV of those keys.

    Rows of the same (b, h) are evaluated together through one matrix
    product; rows remain independent.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if do is not None:
        do = _f64(do)
    B, n, hq, d = q.shape
    nk, hkv = k.shape[1], k.shape[2]
    rows = [tuple(int(x) for x in r) for r in rows]
    R = len(rows)
    out = {"O": np.zeros((R, d)), "LSE": np.full(R, NEG_INF)}
    if do is not None:
        out["D"] = np.zeros(R)
        out["dQ"] = np.zeros((R, d))
    kv_grads = {}
    by_head = {}
    for idx, (b, h, i) in enumerate(rows):
        by_head.setdefault((b, h), []).append((idx, i))
    for (b, h), items in by_head.items():
        g = _kv_head(h, hq, hkv)
        idxs = np.array([t[0] for t in items])
        ii = np.array([t[1] for t in items])
        kk, vv = k[b, :, g], v[b, :, g]
        s = scale * (q[b, ii, h] @ kk.T)
        if causal:
            s = np.where(np.arange(nk)[None, :] <= ii[:, None], s, NEG_INF)
        lse = _row_lse(s)
        ok = np.isfinite(lse)
        P = np.zeros_like(s)
        P[ok] = np.exp(s[ok] - lse[ok, None])
        o = P @ vv
        out["O"][idxs] = o
        out["LSE"][idxs] = lse
        if do is None:
            continue
        dor = do[b, ii, h]
        D = (dor * o).sum(axis=1)
        dP = dor @ vv.T
        dS = P * (dP - D[:, None])
        out["D"][idxs] = D
        out["dQ"][idxs] = scale * (dS @ kk)
        if want_kv_grads:
            dk_acc, dv_acc = kv_grads.setdefault(
                (b, g), (np.zeros((nk, d)), np.zeros((nk, d))))
            dk_acc += scale * (dS.T @ q[b, ii, h])
            dv_acc += P.T @ dor
    if want_kv_grads:
        out["kv_grads"] = kv_grads
    return out


def attention_bwd_by_row_blocks(q, k, v, do, causal, scale, keys=None, want_dq=True, row_block=512,
                                heads=None):
    """The backward of ``attention_bwd`` for sequences too long for N x N
    matrices: the query rows are taken ``row_block`` at a time, and every row
    is still evaluated against all the keys it sees (rows are independent;
    dK and dV are sums over rows, added one block of rows after another).
    Under a causal mask the rows of a block see only keys before the block's
    last row, so the keys after it are not formed at all.

    ``keys``: key rows whose dK, dV are wanted (default all); ``want_dq``:
    also form dQ (needs dP against every visible key); ``heads``: query heads
    to include (default all; dK, dV then hold only their contributions).
    Written with torch fp64 CPU tensors so that the exponentials and products
    run on every host core.  Returns a dict of float64 numpy arrays: O, LSE,
    D (as in ``attention_bwd``), dQ (if wanted; zero for heads left out) and
    dK, dV of shape [B, len(keys), Hkv, d].
    """
    import torch
    t = [torch.as_tensor(np.asarray(x, dtype=np.float64)) for x in (q, k, v, do)]
    q, k, v, do = t
    B, n, hq, d = q.shape
    nk, hkv = k.shape[1], k.shape[2]
    keys = torch.arange(nk) if keys is None else torch.as_tensor(np.asarray(keys, dtype=np.int64))
    all_keys = keys.numel() == nk and bool((keys == torch.arange(nk)).all())
    heads = range(hq) if heads is None else heads
    O = torch.zeros(B, n, hq, d, dtype=torch.float64)
    LSE = torch.full((B, hq, n), NEG_INF, dtype=torch.float64)
    D = torch.zeros(B, hq, n, dtype=torch.float64)
    dQ = torch.zeros(B, n, hq, d, dtype=torch.float64) if want_dq else None
    dK = torch.zeros(B, keys.numel(), hkv, d, dtype=torch.float64)
    dV = torch.zeros(B, keys.numel(), hkv, d, dtype=torch.float64)
    for b in range(B):
        for h in heads:
            g = _kv_head(h, hq, hkv)
            kk, vv = k[b, :, g], v[b, :, g]
            for r0 in range(0, n, row_block):
                r1 = min(n, r0 + row_block)
                kend = min(r1, nk) if causal else nk  # keys any row of the block can see
                sel_pos = torch.nonzero(keys < kend).flatten()
                if not want_dq and sel_pos.numel() == 0:
                    continue
                qc, dc = q[b, r0:r1, h], do[b, r0:r1, h]
                s = scale * (qc @ kk[:kend].T)
                if causal:
                    vis = torch.arange(kend)[None, :] <= torch.arange(r0, r1)[:, None]
                    s = torch.where(vis, s, torch.tensor(NEG_INF, dtype=torch.float64))
                m = s.max(dim=1).values
                ok = torch.isfinite(m)
                lse = torch.full_like(m, NEG_INF)
                lse[ok] = m[ok] + torch.log(torch.exp(s[ok] - m[ok, None]).sum(dim=1))
                P = torch.zeros_like(s)
                P[ok] = torch.exp(s[ok] - lse[ok, None])
                del s
                o = P @ vv[:kend]
                Dr = (dc * o).sum(dim=1)
                O[b, r0:r1, h], LSE[b, h, r0:r1], D[b, h, r0:r1] = o, lse, Dr
                if want_dq or all_keys:
                    dS = P * (dc @ vv[:kend].T - Dr[:, None])
                    if want_dq:
                        dQ[b, r0:r1, h] = scale * (dS @ kk[:kend])
                    if all_keys:
                        dK[b, :kend, g] += scale * (dS.T @ qc)
                        dV[b, :kend, g] += P.T @ dc
                        continue
                    del dS
                if sel_pos.numel():
                    sk = keys[sel_pos]
                    Ps = P[:, sk]
                    dSs = Ps * (dc @ vv[sk].T - Dr[:, None])
                    dK[b, sel_pos, g] += scale * (dSs.T @ qc)
                    dV[b, sel_pos, g] += Ps.T @ dc
    out = {"O": O.numpy(), "LSE": LSE.numpy(), "D": D.numpy(), "dK": dK.numpy(), "dV": dV.numpy()}
    if want_dq:
        out["dQ"] = dQ.numpy()
    return out


# ---------------------------------------------------------------------------
# Blockwise mode: the ring schedule and the rescaled (max, exp_sum,
# weighted_output) merge.  Used to pin the merge algebra against the plain
# definition above, and as the reference for the block/merge entry points.
# ---------------------------------------------------------------------------

def ring_schedule(P, causal):
    """Ring order of "Ring Attention: Partition Sequence Length, Not Batch":
    at step s host i holds the KV chunk of host (i - s) mod P.  Returns, per
    host, the list of chunks it computes against; under a causal mask chunks
    wholly after the host's queries (j > i) are skipped."""
    sched = []
    for i in range(P):
        blocks = [(i - s) % P for s in range(P)]
        if causal:
            blocks = [j for j in blocks if j <= i]
        sched.append(blocks)
    return sched


def block_state(q, k, v, causal, scale, q_off, kv_off, q_pos=None, kv_pos=None):
    """Partial result of one (Q block, KV block) pair as the triple
    (m [B,Hq,Nq], l [B,Hq,Nq], o [B,Nq,Hq,d]):
    m_i = max_j s_ij, l_i = sum_j exp(s_ij - m_i), o_i = sum_j exp(s_ij - m_i) v_j.
    A row with no visible key gives m = -inf, l = 0, o = 0.  Sequence
    positions default to q_off + row and kv_off + row (contiguous blocks);
    q_pos / kv_pos give them explicitly (e.g. striped blocks)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, nq, hq, d = q.shape
    nk, hkv = k.shape[1], k.shape[2]
    vis = _visible(nq, nk, causal, q_off, kv_off, q_pos, kv_pos)
    m = np.full((B, hq, nq), NEG_INF)
    l = np.zeros((B, hq, nq))
    o = np.zeros((B, nq, hq, d))
    for b in range(B):
        for h in range(hq):
            g = _kv_head(h, hq, hkv)
            s = _scores(q[b, :, h], k[b, :, g], scale, vis)
            mm = s.max(axis=1)
            ok = np.isfinite(mm)
            e = np.zeros_like(s)
            e[ok] = np.exp(s[ok] - mm[ok, None])
            m[b, h] = mm
            l[b, h] = e.sum(axis=1)
            o[b, :, h] = e @ v[b, :, g]
    return m, l, o


def merge_states(a, b):
    """Merge two triples: m = max(m_a, m_b); each side is rescaled by
    exp(m_side - m) before summing l and o.  A side with m = -inf (nothing
    seen) gets weight 0."""
    ma, la, oa = (_f64(x) for x in a)
    mb, lb, ob = (_f64(x) for x in b)
    m = np.maximum(ma, mb)
    fin = np.isfinite(m)
    wa = np.zeros_like(m)
    wb = np.zeros_like(m)
    wa[fin] = np.where(np.isfinite(ma[fin]), np.exp(ma[fin] - m[fin]), 0.0)
    wb[fin] = np.where(np.isfinite(mb[fin]), np.exp(mb[fin] - m[fin]), 0.0)
    l = wa * la + wb * lb
    # weights are [B, H, N]; o is [B, N, H, d]
    wa_o = np.transpose(wa, (0, 2, 1))[..., None]
    wb_o = np.transpose(wb, (0, 2, 1))[..., None]
    o = wa_o * oa + wb_o * ob
    return m, l, o


def finalize_state(state):
    """O = o / l and LSE = m + log l; a row with l = 0 gives O = 0, LSE = -inf."""
    m, l, o = (_f64(x) for x in state)
    ok = l > 0
    LSE = np.full_like(m, NEG_INF)
    LSE[ok] = m[ok] + np.log(l[ok])
    inv = np.zeros_like(l)
    inv[ok] = 1.0 / l[ok]
    O = o * np.transpose(inv, (0, 2, 1))[..., None]
    return O, LSE


def striped_positions(N, P):
    """Striped layout (load-balanced causal ordering, "Striped Attention" named
    on "Ring Attention: Train 1M Tokens on 8GB GPUs in 2026", comparison
    section): row r of a striped tensor, in host h = r // S at local row
    l = r % S, holds sequence position l * P + h."""
    if N % P:
        raise ValueError("P must divide N")
    S = N // P
    r = np.arange(N)
    return (r % S) * P + r // S


def ring_fwd_blocked_striped(q, k, v, P, scale):
    """Causal forward of the ring on a striped layout: q, k, v are given in
    striped row order; host i holds rows [iS, (i+1)S) (sequence positions
    l * P + i) and merges its queries' partial results against every KV chunk
    in ring order (i - s) mod P.  Returns O, LSE in the same striped order."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, n, hq, d = q.shape
    S = n // P
    pos = striped_positions(n, P)
    O = np.zeros((B, n, hq, d))
    LSE = np.full((B, hq, n), NEG_INF)
    for i, blocks in enumerate(ring_schedule(P, False)):
        qi = q[:, i * S:(i + 1) * S]
        acc = (np.full((B, hq, S), NEG_INF), np.zeros((B, hq, S)), np.zeros((B, S, hq, d)))
        for j in blocks:
            part = block_state(qi, k[:, j * S:(j + 1) * S], v[:, j * S:(j + 1) * S], True, scale, 0, 0,
                               q_pos=pos[i * S:(i + 1) * S], kv_pos=pos[j * S:(j + 1) * S])
            acc = merge_states(acc, part)
        Oi, Li = finalize_state(acc)
        O[:, i * S:(i + 1) * S] = Oi
        LSE[:, :, i * S:(i + 1) * S] = Li
    return O, LSE


def varlen_rows(N, P, host_len):
    """Rows holding real tokens when host i of P (S = N/P rows each) has only
    its first host_len[i] rows valid and the rest is padding ("FAQ" of "Ring
    Attention: Train 1M Tokens on 8GB GPUs in 2026": each host tracks which
    positions are valid and masks the scores instead of computing on padding).
    The valid rows, in order, are the sequence."""
    S = N // P
    return np.concatenate([np.arange(i * S, i * S + int(host_len[i])) for i in range(P)]).astype(np.int64)


def attention_varlen(q, k, v, do, P, host_len, causal, scale):
    """Exact attention (and, with dO given, its gradients) over the valid rows
    only; padded rows get O = 0, LSE = -inf and zero gradients.  Returns
    (O, LSE) or (dQ, dK, dV, O, LSE) in the padded layout.  With no valid row
    at all every row is padding."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, hq, d = q.shape
    rows = varlen_rows(N, P, host_len)
    O = np.zeros_like(q)
    LSE = np.full((B, hq, N), NEG_INF)
    if rows.size == 0:
        if do is None:
            return O, LSE
        return np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), O, LSE
    if do is None:
        Ov, Lv = attention_fwd(q[:, rows], k[:, rows], v[:, rows], causal, scale)
        O[:, rows] = Ov
        LSE[:, :, rows] = Lv
        return O, LSE
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    gq, gk, gv, Ov, Lv, _ = attention_bwd(q[:, rows], k[:, rows], v[:, rows], _f64(do)[:, rows], causal, scale)
    O[:, rows], LSE[:, :, rows] = Ov, Lv
    dq[:, rows], dk[:, rows], dv[:, rows] = gq, gk, gv
    return dq, dk, dv, O, LSE


def ring_fwd_blocked(q, k, v, P, causal, scale):
    """Forward pass as the ring computes it: host i starts from the empty
    triple and, in ring order, merges the partial result of its queries
    against each KV chunk it holds; finally divides by the denominator."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, n, hq, d = q.shape
    if n % P:
        raise ValueError("P must divide N")
    S = n // P
    O = np.zeros((B, n, hq, d))
    LSE = np.full((B, hq, n), NEG_INF)
    for i, blocks in enumerate(ring_schedule(P, causal)):
        qi = q[:, i * S:(i + 1) * S]
        acc = (np.full((B, hq, S), NEG_INF), np.zeros((B, hq, S)),
               np.zeros((B, S, hq, d)))
        for j in blocks:
            part = block_state(qi, k[:, j * S:(j + 1) * S], v[:, j * S:(j + 1) * S],
                               causal, scale, i * S, j * S)
            acc = merge_states(acc, part)
        Oi, Li = finalize_state(acc)
        O[:, i * S:(i + 1) * S] = Oi
        LSE[:, :, i * S:(i + 1) * S] = Li
    return O, LSE
