"""Seeded synthetic inputs for the attention workloads.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both the CUDA path (through the tests and the
benchmark) and the fp64 oracle can consume what it produces.

Workloads (B, N, heads, head dim, virtual hosts P):
  1  fp32 non-causal, B=1, H=2, N=512, d=64, P=4; forward + backward
  2  bf16 causal forward, B=1, H=16, N=32768, d=128, P=8
  3  bf16 causal forward + backward, B=1, H=16, N=131072, d=128, P=32
  4  bf16 causal grouped-query, B=1, Hq=32, Hkv=8, N=262144, d=128, P=32;
     Q ~ 4 N(0,1) (logits reach about +-30), 1% of V entries set to +-50
  5  bf16 causal forward + backward, B=1, H=32, N=1048576, d=128, P=64
Q, K, V, dO ~ N(0,1) in fp32 rounded to the working dtype; the seed of
workload c is 1000 + c.
"""
import torch

WORKLOADS = {
    1: dict(name="fp32 non-causal B1 H2 N512 d64 P4", B=1, N=512, Hq=2, Hkv=2, d=64, P=4,
            causal=False, dtype=torch.float32, bwd=True, q_scale=1.0, v_outlier_frac=0.0),
    2: dict(name="bf16 causal B1 H16 N32768 d128 P8", B=1, N=32768, Hq=16, Hkv=16, d=128, P=8,
            causal=True, dtype=torch.bfloat16, bwd=False, q_scale=1.0, v_outlier_frac=0.0),
    3: dict(name="bf16 causal B1 H16 N131072 d128 P32", B=1, N=131072, Hq=16, Hkv=16, d=128,
            P=32, causal=True, dtype=torch.bfloat16, bwd=True, q_scale=1.0, v_outlier_frac=0.0),
    4: dict(name="bf16 causal GQA B1 Hq32 Hkv8 N262144 d128 P32", B=1, N=262144, Hq=32, Hkv=8,
            d=128, P=32, causal=True, dtype=torch.bfloat16, bwd=True, q_scale=4.0,
            v_outlier_frac=0.01),
    5: dict(name="bf16 causal B1 H32 N1048576 d128 P64", B=1, N=1048576, Hq=32, Hkv=32, d=128,
            P=64, causal=True, dtype=torch.bfloat16, bwd=True, q_scale=1.0, v_outlier_frac=0.0),
}
V_OUTLIER = 50.0
CHUNK_ROWS = 8192


def _fill(out, gen, scale=1.0, outlier_frac=0.0):
    """Fill out [B, N, H, d] with N(0,1)*scale drawn in fp32 (row chunks), then
    optionally replace a Bernoulli(outlier_frac) subset by +-50."""
    B, N, H, d = out.shape
    for b in range(B):
        for r0 in range(0, N, CHUNK_ROWS):
            r1 = min(N, r0 + CHUNK_ROWS)
            x = torch.randn((r1 - r0, H, d), generator=gen, device=out.device, dtype=torch.float32)
            if scale != 1.0:
                x.mul_(scale)
            if outlier_frac > 0.0:
                hit = torch.rand(x.shape, generator=gen, device=out.device) < outlier_frac
                sign = torch.where(torch.rand(x.shape, generator=gen, device=out.device) < 0.5,
                                   -V_OUTLIER, V_OUTLIER)
                x = torch.where(hit, sign, x)
            out[b, r0:r1].copy_(x)
    return out


def make_tensors(B, N, Hq, Hkv, d, dtype, device, seed, q_scale=1.0, v_outlier_frac=0.0,
                 with_do=True, N_kv=None):
    """Seeded q [B,N,Hq,d], k, v [B,N_kv,Hkv,d], dO [B,N,Hq,d] in `dtype`."""
    N_kv = N if N_kv is None else N_kv
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q = _fill(torch.empty(B, N, Hq, d, dtype=dtype, device=device), gen, q_scale)
    k = _fill(torch.empty(B, N_kv, Hkv, d, dtype=dtype, device=device), gen)
    v = _fill(torch.empty(B, N_kv, Hkv, d, dtype=dtype, device=device), gen, 1.0, v_outlier_frac)
    do = _fill(torch.empty(B, N, Hq, d, dtype=dtype, device=device), gen) if with_do else None
    return q, k, v, do


def make_config(cid, device, with_do=None):
    c = WORKLOADS[cid]
    if with_do is None:
        with_do = c["bwd"]
    return make_tensors(c["B"], c["N"], c["Hq"], c["Hkv"], c["d"], c["dtype"], device,
                        1000 + cid, c["q_scale"], c["v_outlier_frac"], with_do)


def sample_rows(cid, n_random=512, heads=None, tail=512, seed=None):
    """Seeded query rows (b, h, i) for checking a large workload row by row:
    n_random uniform rows drawn from `heads` (default: all), plus row 0, row
    N-1 and the first/last rows of several hosts and 128-row tiles, plus the
    last `tail` rows of one seeded head (which, under a causal mask, are the
    only rows that see the last `tail` keys)."""
    c = WORKLOADS[cid]
    N, Hq, P = c["N"], c["Hq"], c["P"]
    S = N // P
    g = torch.Generator().manual_seed(7000 + cid if seed is None else seed)
    heads = list(range(Hq)) if heads is None else list(heads)
    hsel = torch.tensor(heads)[torch.randint(len(heads), (n_random,), generator=g)]
    isel = torch.randint(N, (n_random,), generator=g)
    rows = {(0, int(h), int(i)) for h, i in zip(hsel, isel)}
    hosts = sorted({0, 1, P // 2, P - 1})
    for hst in hosts:
        h = heads[hst % len(heads)]
        for i in (hst * S, hst * S + 127, hst * S + 128, (hst + 1) * S - 1):
            rows.add((0, h, min(i, N - 1)))
    rows.add((0, heads[0], 0))
    rows.add((0, heads[-1], N - 1))
    tail_head = heads[int(torch.randint(len(heads), (1,), generator=g))]
    rows = sorted(rows)
    tail_rows = [(0, tail_head, i) for i in range(N - tail, N)] if tail else []
    return rows, tail_rows, tail_head


def make_ffn(T, d_model, d_hidden, dtype, device, seed):
    """Seeded synthetic feed-forward inputs: x, dy ~ N(0, 1); W1 ~ N(0, 1/d_model),
    W2 ~ N(0, 1/d_hidden) (unit-variance activations through both layers), each
    drawn in fp32 and rounded to dtype."""
    g = torch.Generator(device=device).manual_seed(seed)

    def draw(shape, std):
        return (torch.randn(shape, generator=g, dtype=torch.float32, device=device) * std).to(dtype)

    x = draw((T, d_model), 1.0)
    w1 = draw((d_hidden, d_model), d_model ** -0.5)
    w2 = draw((d_model, d_hidden), d_hidden ** -0.5)
    dy = draw((T, d_model), 1.0)
    return x, w1, w2, dy

