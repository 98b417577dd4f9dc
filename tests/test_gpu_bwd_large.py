"""Backward pass at the full 128K GQA causal size, in the launch configuration
`bench.py --pass bwd --workload bf16_128k_gqa_causal` times (16 zigzag chunks
walked in ring order): sampled dQ rows and sampled dK, dV key rows against
the fp64 definition (each exact against every visible (query, key) pair that
contributes to it), and every gradient element through chunking invariance
against a one-chunk run ("Ring Attention: Distributed Reads with Online
Softmax", section "Backward must aggregate shared dependencies": the
distributed gradients must match a single-device reference).

Tolerance as in tests/test_gpu_bwd.py: max|err| <= 1e-2 * max|ref| per
gradient (P and dS are rounded to bf16 before their products).
"""
import numpy as np
import pytest
import torch

from blockwise_attention_online_gb300 import (device_status, layouts, ring_attention,
                                              ring_attention_bwd, workloads)
from _util import f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 1e-2


def _normwise(name, got, ref):
    err = (got - ref).abs().max().item()
    scale = max(ref.abs().max().item(), 1e-6)
    assert err <= TOL * scale, f"{name}: max-abs {err:.3e} vs {TOL} x {scale:.3e}"


def test_bwd_128k_gqa_zigzag_sampled_rows_and_invariance():
    w = workloads.WORKLOADS["bf16_128k_gqa_causal"]
    q, k, v = workloads.make_qkv(w, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(99)
    do = torch.randn(q.shape, device=DEV, generator=g).to(torch.bfloat16)
    P, kind, S = w.n_chunks, w.layout, w.S
    rs = layouts.rank_spans(kind, S, P)
    kc = [t.contiguous() for t in layouts.shard(k, kind, P)]
    vc = [t.contiguous() for t in layouts.shard(v, kind, P)]
    qs = torch.cat(layouts.shard(q, kind, P), dim=2).contiguous()
    dos = torch.cat(layouts.shard(do, kind, P), dim=2).contiguous()
    segs = [(S // P, s) for s in rs]
    O, m, l = ring_attention(qs, kc, vc, chunk_spans=rs, q_segments=segs, causal=True)
    dq, dk, dv = ring_attention_bwd(qs, kc, vc, O, dos, m, l, chunk_spans=rs, q_segments=segs,
                                    causal=True)
    device_status()
    del O, qs, dos
    dq = layouts.to_global(dq, kind, P)
    dk = layouts.to_global(torch.cat(dk, dim=2), kind, P)
    dv = layouts.to_global(torch.cat(dv, dim=2), kind, P)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()

    # sampled dQ rows of two query heads (of different key/value heads)
    group = w.Hq // w.Hkv
    half = S // (2 * P)
    rows = [0, 1, half - 1, half, S // 2 - 1, S // 2, S - half - 1, S - half, S - 1]
    rows += [int(x) for x in np.random.default_rng(5).integers(0, S, size=6)]
    refs, gots = [], []
    for h in (0, 29):
        kh, vh = f64(k[0, h // group]), f64(v[0, h // group])
        qh, doh = f64(q[0, h]), f64(do[0, h])
        for i in rows:
            s = (qh[i] @ kh[: i + 1].T) * w.scale
            p = np.exp(s - s.max())
            p /= p.sum()
            dp = doh[i] @ vh[: i + 1].T
            ds = p * (dp - (p * dp).sum())
            refs.append((ds @ kh[: i + 1]) * w.scale)
            gots.append(f64(dq[0, h, i]))
    refs, gots = np.stack(refs), np.stack(gots)
    err = np.abs(gots - refs).max()
    assert err <= TOL * np.abs(refs).max(), f"sampled dq rows: max-abs {err:.3e}"

    # sampled key rows of dK and dV of key/value head 0 (query heads 0..3),
    # from the last 2048 positions: with the causal mask exactly the query
    # rows [S - 2048, S) see them, so each is exact against all of its terms
    tail = 2048
    keys = sorted({S - 1, S - 2, S - tail, S - tail + 1, S - tail // 2}
                  | {int(x) for x in np.random.default_rng(6).integers(S - tail, S, size=6)})
    kh, vh = f64(k[0, 0]), f64(v[0, 0])
    ref_dk = np.zeros((len(keys), w.D))
    ref_dv = np.zeros((len(keys), w.D))
    kpos = np.arange(S)
    for h in range(group):
        qh, doh = f64(q[0, h]), f64(do[0, h])
        for r0 in range(S - tail, S, 256):
            r1 = min(S, r0 + 256)
            sc = (qh[r0:r1] @ kh.T) * w.scale
            sc[kpos[None, :] > np.arange(r0, r1)[:, None]] = -np.inf
            pm = np.exp(sc - sc.max(axis=1, keepdims=True))
            pm /= pm.sum(axis=1, keepdims=True)
            delta = (doh[r0:r1] * (pm @ vh)).sum(axis=1)
            pk = pm[:, keys]
            ds = pk * (doh[r0:r1] @ vh[keys].T - delta[:, None])
            ref_dv += pk.T @ doh[r0:r1]
            ref_dk += w.scale * (ds.T @ qh[r0:r1])
    for name, got, ref in (("sampled dk rows", dk[0, 0, keys], ref_dk),
                           ("sampled dv rows", dv[0, 0, keys], ref_dv)):
        err = np.abs(f64(got) - ref).max()
        assert err <= TOL * np.abs(ref).max(), f"{name}: max-abs {err:.3e}"

    # every element against a one-chunk run of the same problem
    O1, m1, l1 = ring_attention(q, [k], [v], causal=True)
    dq1, dk1, dv1 = ring_attention_bwd(q, [k], [v], O1, do, m1, l1, causal=True)
    device_status()
    _normwise("dq", dq, dq1)
    _normwise("dk", dk, dk1[0])
    _normwise("dv", dv, dv1[0])
