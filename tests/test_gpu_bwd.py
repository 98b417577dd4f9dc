"""Parity of the backward pass (ra_ring_attention_bwd) with the fp64 oracle.

The oracle (oracle.backward.attention_backward) differentiates O by the
definition; the library recomputes the probability tiles per chunk from the
forward's m, l ("Ring Attention: Distributed Reads with Online Softmax",
section "Backward must aggregate shared dependencies") and sums each chunk's
dK, dV over every query row.

Tolerance (no page states one): P and dS are rounded to bf16 before their
products (relative error at most 2^-8 each), products accumulate in fp32.
Normwise, the error of each gradient stays within 1e-2 of the reference's
largest magnitude; the tests check max|err| <= 1e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from blockwise_attention_online_gb300 import device_status, layouts, ring_attention, ring_attention_bwd
from _util import f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 1e-2


def _inputs(seed, B, Hq, Hkv, S, D, Sq=None):
    g = torch.Generator(device="cpu").manual_seed(seed)
    Sq = S if Sq is None else Sq
    q = torch.randn(B, Hq, Sq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    do = torch.randn(B, Hq, Sq, D, generator=g).to(torch.bfloat16)
    return q, k, v, do


def _check(name, got, ref):
    got, ref = f64(got), np.asarray(ref, dtype=np.float64)
    assert not np.isnan(got).any(), f"{name}: NaN"
    err = np.abs(got - ref).max()
    scale = max(np.abs(ref).max(), 1e-6)
    assert err <= TOL * scale, f"{name}: max-abs {err:.3e} vs {TOL} x {scale:.3e}"


def _layout_bwd(q, k, v, do, kind, P, causal, out_dtype=None):
    """Forward + backward on per-rank shards; gradients back in global order."""
    S = k.shape[2]
    rs = layouts.rank_spans(kind, S, P)
    kc = [t.contiguous().to(DEV) for t in layouts.shard(k, kind, P)]
    vc = [t.contiguous().to(DEV) for t in layouts.shard(v, kind, P)]
    qs = torch.cat(layouts.shard(q, kind, P), dim=2).contiguous().to(DEV)
    dos = torch.cat(layouts.shard(do, kind, P), dim=2).contiguous().to(DEV)
    segs = [(S // P, s) for s in rs]
    O, m, l = ring_attention(qs, kc, vc, chunk_spans=rs, q_segments=segs, causal=causal,
                             out_dtype=out_dtype)
    if out_dtype is not None:
        dos = dos.contiguous()
    dq, dk, dv = ring_attention_bwd(qs, kc, vc, O, dos, m, l, chunk_spans=rs, q_segments=segs,
                                    causal=causal)
    torch.cuda.synchronize()
    device_status()
    dq = layouts.to_global(dq.cpu(), kind, P)
    dk = torch.cat([t.cpu() for t in dk], dim=2)
    dv = torch.cat([t.cpu() for t in dv], dim=2)
    order = np.concatenate([np.asarray(r) for r in oracle.layouts.LAYOUTS[kind](S, P)])
    inv = np.argsort(order)
    return dq, dk[:, :, inv], dv[:, :, inv]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,kind,P,causal", [
    (1, 2, 2, 512, 128, "contiguous", 4, False),
    (1, 4, 2, 768, 128, "zigzag", 2, True),
    (2, 2, 1, 640, 64, "striped", 4, True),
    (1, 8, 2, 1024, 128, "contiguous", 8, True),
    (1, 4, 2, 640, 96, "zigzag", 2, True),
    (2, 2, 2, 384, 96, "contiguous", 3, False),
])
def test_backward_matches_oracle(B, Hq, Hkv, S, D, kind, P, causal):
    q, k, v, do = _inputs(11, B, Hq, Hkv, S, D)
    dq, dk, dv = _layout_bwd(q, k, v, do, kind, P, causal)
    pos = np.arange(S)
    rq, rk, rv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), pos, pos, causal,
                                           D ** -0.5)
    _check("dq", dq, rq)
    _check("dk", dk, rk)
    _check("dv", dv, rv)


def test_backward_ragged_rows_and_chunks():
    """Sq not a multiple of 128, chunks of uneven, non-multiple-of-128 lengths."""
    q, k, v, do = _inputs(12, 1, 2, 1, 700, 128, Sq=333)
    lens = [1, 200, 99, 400]
    kc = [t.contiguous().to(DEV) for t in torch.split(k, lens, dim=2)]
    vc = [t.contiguous().to(DEV) for t in torch.split(v, lens, dim=2)]
    # queries at positions 367..699 (the end of the key sequence), causal
    qpos0 = 700 - 333
    segs = [(333, [(333, qpos0, 1)])]
    qd, dod = q.to(DEV), do.to(DEV)
    O, m, l = ring_attention(qd, kc, vc, q_segments=segs, causal=True)
    dq, dk, dv = ring_attention_bwd(qd, kc, vc, O, dod, m, l, q_segments=segs, causal=True)
    torch.cuda.synchronize()
    device_status()
    rq, rk, rv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do),
                                           np.arange(qpos0, 700), np.arange(700), True, 128 ** -0.5)
    _check("dq", dq, rq)
    _check("dk", torch.cat([t.cpu() for t in dk], dim=2), rk)
    _check("dv", torch.cat([t.cpu() for t in dv], dim=2), rv)


def test_backward_with_fp32_output_and_unseen_chunk():
    """O kept in fp32; a chunk that lies entirely after every query gets zero
    gradients."""
    q, k, v, do = _inputs(13, 1, 2, 2, 512, 64, Sq=256)
    kc = [k[:, :, :256].contiguous().to(DEV), k[:, :, 256:].contiguous().to(DEV)]
    vc = [v[:, :, :256].contiguous().to(DEV), v[:, :, 256:].contiguous().to(DEV)]
    qd, dod = q.to(DEV), do.to(DEV)
    O, m, l = ring_attention(qd, kc, vc, causal=True, out_dtype=torch.float32)
    dq, dk, dv = ring_attention_bwd(qd, kc, vc, O, dod, m, l, causal=True)
    torch.cuda.synchronize()
    device_status()
    rq, rk, rv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), np.arange(256),
                                           np.arange(512), True, 64 ** -0.5)
    _check("dq", dq, rq)
    _check("dk", dk[0], rk[:, :, :256])
    _check("dv", dv[0], rv[:, :, :256])
    assert float(dk[1].abs().max()) == 0.0 and float(dv[1].abs().max()) == 0.0


def test_backward_chunking_invariance_at_8k():
    """The 8K workload's shape (8 heads, 8192 keys, head_dim 128): eight ring
    chunks against one chunk; the recomputed tiles differ only in rounding."""
    q, k, v, do = _inputs(14, 1, 8, 8, 8192, 128)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    O, m, l = ring_attention(qd, [kd], [vd], causal=True)
    dq1, dk1, dv1 = ring_attention_bwd(qd, [kd], [vd], O, dod, m, l, causal=True)
    kc = list(torch.split(kd, 1024, dim=2))
    vc = list(torch.split(vd, 1024, dim=2))
    kc = [t.contiguous() for t in kc]
    vc = [t.contiguous() for t in vc]
    dq8, dk8, dv8 = ring_attention_bwd(qd, kc, vc, O, dod, m, l, causal=True)
    torch.cuda.synchronize()
    device_status()
    for a, b in ((dq8, dq1), (torch.cat(dk8, dim=2), dk1[0]), (torch.cat(dv8, dim=2), dv1[0])):
        assert torch.isfinite(a).all()
        # identical arithmetic per tile: the same values
        assert torch.equal(a, b)
    # sampled query rows of dQ against the oracle (head 3, rows across the sequence)
    rows = [0, 1, 127, 128, 4095, 4096, 8191]
    h = 3
    qh, kh, vh, doh = (f64(t[0, h]) for t in (q, k, v, do))
    refs, gots = [], []
    for i in rows:
        s = (qh[i] @ kh[: i + 1].T) * 128 ** -0.5
        p = np.exp(s - s.max())
        p /= p.sum()
        dp = doh[i] @ vh[: i + 1].T
        ds = p * (dp - (p * dp).sum())
        refs.append((ds @ kh[: i + 1]) * 128 ** -0.5)   # row 0 sees one key: exactly 0
        gots.append(f64(dq1[0, h, i]))
    _check("sampled dq rows", np.stack(gots), np.stack(refs))
