"""Helpers shared by the parity tests: tolerances and comparisons against the
fp64 oracle.  The tolerances are the stated ones: fp32 inputs max |err| <= 1e-4
on every output; 16-bit inputs with fp32 accumulation max |err| <= 2e-2 and
mean |err| <= 2e-3 on O, dQ, dK, dV and max |err| <= 1e-3 on LSE."""
import numpy as np
import torch

TOL = {
    torch.float32: dict(max=1e-4, mean=None, lse=1e-4),
    torch.bfloat16: dict(max=2e-2, mean=2e-3, lse=1e-3),
    torch.float16: dict(max=2e-2, mean=2e-3, lse=1e-3),
}


def f64(t):
    """Exact values of a device tensor as float64 (bf16/fp16 -> fp32 is exact)."""
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def check(name, got, want, dtype, kind="out"):
    tol = TOL[dtype]
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{name}: shape {got.shape} vs {want.shape}"
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), f"{name}: non-finite pattern differs"
    assert np.array_equal(got[~fin], want[~fin]), f"{name}: infinite entries differ"
    err = np.abs(got[fin] - want[fin])
    if err.size == 0:
        return 0.0
    lim = tol["lse"] if kind == "lse" else tol["max"]
    assert err.max() <= lim, f"{name}: max |err| {err.max():.3e} > {lim:g}"
    if kind != "lse" and tol["mean"] is not None:
        assert err.mean() <= tol["mean"], f"{name}: mean |err| {err.mean():.3e} > {tol['mean']:g}"
    return float(err.max())


def state_view(m, l, o):
    """What a (m, l, o) state represents: o / l and m + log(l) (any reference
    point m gives the same pair)."""
    m, l, o = (np.asarray(x, dtype=np.float64) for x in (m, l, o))
    ok = l > 0
    lse = np.full_like(m, -np.inf)
    lse[ok] = m[ok] + np.log(l[ok])
    inv = np.where(ok, 1.0 / np.where(ok, l, 1.0), 0.0)
    return o * np.transpose(inv, (0, 2, 1))[..., None], lse
