"""Backward pass checked element by element against the fp64 definition.

The kernel is given the oracle's own forward results (O in fp32, m, l), so
that every input of the comparison comes from the definition, and each
gradient element is compared with the oracle's within the rounding bound of
the kernel's arithmetic ("Ring Attention: Distributed Reads with Online
Softmax", section "Backward must aggregate shared dependencies": check the
gradients against a single-device reference).

Bound (oracle.gradient_rounding_bounds): P and dS are rounded to bf16 (unit
roundoff 2^-8) before their products, which accumulate in fp32, so

    |dV - dV_ref| <= 2^-8 P^T |dO|,
    |dQ - dQ_ref| <= scale 2^-8 |dS| |K|,  |dK - dK_ref| <= scale 2^-8 |dS|^T |Q|;

the tests allow twice that (the fp32 parts add errors about a thousand times
smaller) plus 1e-6 of the gradient's largest magnitude.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from blockwise_attention_online_gb300 import device_status, layouts, ring_attention_bwd
from _util import f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed, B, Hq, Hkv, S, D, Sq=None):
    g = torch.Generator(device="cpu").manual_seed(seed)
    Sq = S if Sq is None else Sq
    q = torch.randn(B, Hq, Sq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    do = torch.randn(B, Hq, Sq, D, generator=g).to(torch.bfloat16)
    return q, k, v, do


def _assert_within(name, got, ref, bound):
    got, ref = f64(got), np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), f"{name}: not finite"
    err = np.abs(got - ref)
    tol = 2.0 * bound + 1e-6 * max(np.abs(ref).max(), 1e-30)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} elements outside the bound; worst at {i}: "
                             f"got {got[i]:.6e} want {ref[i]:.6e} bound {tol[i]:.3e}")
    return float((err / np.maximum(tol, 1e-300)).max())


def _oracle_forward(q, k, v, qpos, kpos, causal, scale, docs=None):
    O, m, l = oracle.full_attention(f64(q), f64(k), f64(v), qpos, kpos, causal, scale, docs)
    return (torch.from_numpy(O).float(), torch.from_numpy(m).float(), torch.from_numpy(l).float())


@pytest.mark.parametrize("B,Hq,Hkv,S,D,kind,P,causal", [
    (1, 2, 2, 512, 128, "contiguous", 4, False),
    (1, 4, 2, 768, 128, "zigzag", 2, True),
    (2, 2, 1, 640, 64, "striped", 4, True),
    (1, 4, 2, 640, 96, "zigzag", 2, True),
    (1, 8, 2, 1024, 128, "contiguous", 8, True),
    # more tile CTAs (96 key tiles, 96 query tiles) than SMs: several waves
    (1, 4, 4, 3072, 64, "zigzag", 4, True),
])
def test_gradients_within_rounding_bound(B, Hq, Hkv, S, D, kind, P, causal):
    q, k, v, do = _inputs(41, B, Hq, Hkv, S, D)
    scale = 1 / math.sqrt(D)
    pos = np.arange(S)
    O, m, l = _oracle_forward(q, k, v, pos, pos, causal, scale)
    rs = layouts.rank_spans(kind, S, P)
    kc = [t.contiguous().to(DEV) for t in layouts.shard(k, kind, P)]
    vc = [t.contiguous().to(DEV) for t in layouts.shard(v, kind, P)]
    shard_q = lambda t: torch.cat(layouts.shard(t, kind, P), dim=2).contiguous().to(DEV)
    qs, dos, Os = shard_q(q), shard_q(do), shard_q(O)
    ms = shard_q(m.unsqueeze(-1)).squeeze(-1).contiguous()
    ls = shard_q(l.unsqueeze(-1)).squeeze(-1).contiguous()
    segs = [(S // P, s) for s in rs]
    dq, dk, dv = ring_attention_bwd(qs, kc, vc, Os, dos, ms, ls, chunk_spans=rs, q_segments=segs,
                                    causal=causal)
    device_status()
    dq = layouts.to_global(dq.cpu(), kind, P)
    order = np.concatenate([np.asarray(r) for r in oracle.layouts.LAYOUTS[kind](S, P)])
    inv = np.argsort(order)
    dk = torch.cat([t.cpu() for t in dk], dim=2)[:, :, inv]
    dv = torch.cat([t.cpu() for t in dv], dim=2)[:, :, inv]
    rq, rk, rv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), pos, pos, causal, scale)
    bq, bk, bv = oracle.gradient_rounding_bounds(f64(q), f64(k), f64(v), f64(do), pos, pos, causal,
                                                 scale)
    _assert_within("dq", dq, rq, bq)
    _assert_within("dk", dk, rk, bk)
    _assert_within("dv", dv, rv, bv)


def test_gradients_ragged_and_documents_within_bound():
    """Ragged query and key tiles, uneven chunks, packed documents with a
    causal mask; a chunk no query can see gets exact zeros."""
    S, Sq, D = 700, 333, 128
    q, k, v, do = _inputs(42, 1, 2, 1, S, D, Sq=Sq)
    scale = 1 / math.sqrt(D)
    qpos, kpos = np.arange(S - Sq, S), np.arange(S)
    docs = [0, 5, 300, 301, 420, 700]
    O, m, l = _oracle_forward(q, k, v, qpos, kpos, True, scale, docs)
    lens = [1, 200, 99, 400]
    kc = [t.contiguous().to(DEV) for t in torch.split(k, lens, dim=2)]
    vc = [t.contiguous().to(DEV) for t in torch.split(v, lens, dim=2)]
    segs = [(Sq, [(Sq, S - Sq, 1)])]
    dq, dk, dv = ring_attention_bwd(q.to(DEV), kc, vc, O.to(DEV), do.to(DEV), m.to(DEV), l.to(DEV),
                                    q_segments=segs, causal=True, docs=docs)
    device_status()
    rq, rk, rv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), qpos, kpos, True, scale,
                                           docs)
    bq, bk, bv = oracle.gradient_rounding_bounds(f64(q), f64(k), f64(v), f64(do), qpos, kpos, True,
                                                 scale, docs)
    _assert_within("dq", dq, rq, bq)
    _assert_within("dk", torch.cat([t.cpu() for t in dk], dim=2), rk, bk)
    _assert_within("dv", torch.cat([t.cpu() for t in dv], dim=2), rv, bv)
