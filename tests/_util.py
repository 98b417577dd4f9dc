"""Shared helpers of the parity tests: tolerances, row samples, layout runs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from blockwise_attention_online_gb300 import layouts, ring_attention

# fp32 path: max-abs 1e-5 on O and m; l (a sum of up to Sk terms of size <= 1)
# to 1e-5 relative once it exceeds 1.
F32_ATOL = 1e-5
# bf16 path: O max-abs 1e-2; m and l relative 1e-3 (for m near 0 the bound is
# 1e-3 absolute, a pure relative bound being ill-posed there).
BF16_O_ATOL = 1e-2
BF16_ML_RTOL = 1e-3


def f64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def _same_inf(a, b):
    ia, ib = np.isinf(a), np.isinf(b)
    assert np.array_equal(ia, ib), "-inf pattern differs"
    assert np.array_equal(np.sign(a[ia]), np.sign(b[ib]))
    return ~ia


def assert_f32(O, m, l, Oref, mref, lref):
    O, m, l = f64(O), f64(m), f64(l)
    assert not np.isnan(O).any() and not np.isnan(l).any()
    err = np.abs(O - Oref).max() if O.size else 0.0
    assert err <= F32_ATOL, f"O max-abs {err:.3e}"
    fin = _same_inf(m, mref)
    if fin.any():
        assert np.abs(m[fin] - mref[fin]).max() <= F32_ATOL
    assert (np.abs(l - lref) <= F32_ATOL * np.maximum(1.0, lref)).all()


def bf16_half_ulp(x):
    """Half a unit in the last place of bfloat16 (8 significant bits) at |x|:
    the rounding a bf16 output carries on top of the computed value."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


# Below this |O| a bf16 output's own rounding (at most 2^-8 there) leaves
# room inside 1e-2, so the plain bound applies; above it half an ulp of the
# reference (2^-7 from |O| = 2, 2^-6 from 4) is allowed on top.
BF16_O_SLACK_FROM = 2.0


def assert_bf16(O, m, l, Oref, mref, lref, what=""):
    """O: within 1e-2 of the oracle when O is fp32, and for a bf16 O wherever
    |O_ref| < 2; a bf16 O at |O_ref| >= 2 may in addition carry its own
    rounding (half an ulp of the reference value)."""
    out_bf16 = isinstance(O, torch.Tensor) and O.dtype == torch.bfloat16
    O, m, l = f64(O), f64(m), f64(l)
    assert not np.isnan(O).any() and not np.isnan(l).any(), f"{what}: NaN"
    slack = np.where(np.abs(Oref) >= BF16_O_SLACK_FROM, bf16_half_ulp(Oref), 0.0)
    tol = BF16_O_ATOL + (slack if out_bf16 else 0.0)
    excess = np.abs(O - Oref) - tol
    err = np.abs(O - Oref).max() if O.size else 0.0
    if O.size and excess.max() > 0:
        idx = np.unravel_index(np.argmax(excess), O.shape)
        raise AssertionError(f"{what}: O max-abs {err:.3e} ({'bf16' if out_bf16 else 'fp32'} out); "
                             f"worst at {idx}: got {O[idx]:.6f} want {Oref[idx]:.6f}")
    fin = _same_inf(m, mref)
    if fin.any():
        dm = np.abs(m[fin] - mref[fin]) / np.maximum(1.0, np.abs(mref[fin]))
        assert dm.max() <= BF16_ML_RTOL, f"{what}: m rel {dm.max():.3e}"
    pos = lref > 0
    if pos.any():
        dl = np.abs(l[pos] - lref[pos]) / lref[pos]
        assert dl.max() <= BF16_ML_RTOL, f"{what}: l rel {dl.max():.3e}"
    assert np.all(l[~pos] == 0)
    return err


def layout_run(q, k, v, P, kind, causal, scale=None, out_dtype=None, docs=None):
    """Shard global-order q, k, v per ``kind`` over P virtual ranks, run the
    library's ring kernel, return O, m, l back in global order."""
    S = k.shape[2]
    rs = layouts.rank_spans(kind, S, P)
    kc = layouts.shard(k, kind, P)
    vc = layouts.shard(v, kind, P)
    qs = torch.cat(layouts.shard(q, kind, P), dim=2).contiguous()
    segs = [(S // P, s) for s in rs]       # as many segments as chunks: ring order
    O, m, l = ring_attention(qs, kc, vc, chunk_spans=rs, q_segments=segs, causal=causal,
                             scale=scale, out_dtype=out_dtype, docs=docs)
    O = layouts.to_global(O, kind, P)
    m = layouts.to_global(m.unsqueeze(-1), kind, P).squeeze(-1)
    l = layouts.to_global(l.unsqueeze(-1), kind, P).squeeze(-1)
    return O, m, l


def sample_rows(S, boundaries, n_random, seed=1234, tile=128, max_tiles=64):
    """Row sample: first/second/last rows, +-1 around every given boundary and
    around (up to ``max_tiles`` evenly spread) tile boundaries, plus random
    rows drawn with ``seed``."""
    rows = {0, 1, S - 1}
    for bd in boundaries:
        for d in (-1, 0, 1):
            if 0 <= bd + d < S:
                rows.add(bd + d)
    tb = list(range(tile, S, tile))
    if len(tb) > max_tiles:
        tb = tb[:: max(1, len(tb) // max_tiles)]
    for bd in tb:
        for d in (-1, 0):
            rows.add(bd + d)
    rng = np.random.default_rng(seed)
    rows.update(int(x) for x in rng.integers(0, S, size=n_random))
    return sorted(rows)


class LazyHeads:
    """Read-only view handing the oracle one (batch, head) slice at a time as a
    float32 host array, so that device tensors of long sequences never have to
    be copied to the host whole."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        return self.t[idx].float().cpu().numpy()


def oracle_rows(q, k, v, causal, scale, heads, rows, docs=None):
    """fp64 oracle on sampled (head, row) pairs of global-order q, k, v."""
    q, k, v = LazyHeads(q), LazyHeads(k), LazyHeads(v)
    S = k.shape[2]
    pos = np.arange(S)
    trip = [(0, h, i) for h in heads for i in rows]
    O, M, L = oracle.attention_rows(q, k, v, np.arange(q.shape[2]), pos, causal, scale, trip,
                                    docs=docs)
    n = len(rows)
    return (O.reshape(len(heads), n, -1), M.reshape(len(heads), n), L.reshape(len(heads), n))
