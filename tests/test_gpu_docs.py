"""Parity of packed documents (variable-length sequences) with the oracle.

Documents are ranges of global positions [b_d, b_{d+1}); a query sees only
keys of its own document, with the causal rule of "Ring Attention:
Distributed Reads with Online Softmax", section "Causal masks depend on
global positions", on top. The oracle's document mask is pinned on the CPU
(tests/test_oracle_docs.py); here the CUDA path (bf16 tcgen05 kernel, fp32
kernel, chunk statistics, host-buffer entry, backward) is compared with it
under the tolerances of the other parity tests. Boundaries are drawn by
workloads.packed_documents (seeded) and include documents of one position,
boundaries inside 128-row tiles and documents spanning many tiles.
"""
import numpy as np
import pytest
import torch

import oracle
from blockwise_attention_online_gb300 import (chunk_stats, device_status, layouts, ring_attention,
                                              ring_attention_bwd, ring_attention_host, workloads)
from _util import assert_bf16, assert_f32, f64, layout_run, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _qkv(seed, B, Hq, Hkv, S, D, dtype=torch.bfloat16):
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(B, Hq, S, D, generator=g).to(dtype)
    k = torch.randn(B, Hkv, S, D, generator=g).to(dtype)
    v = torch.randn(B, Hkv, S, D, generator=g).to(dtype)
    return q, k, v


def _ref(q, k, v, causal, docs, qpos=None):
    S = k.shape[2]
    qpos = np.arange(q.shape[2]) if qpos is None else qpos
    return oracle.full_attention(f64(q), f64(k), f64(v), qpos, np.arange(S), causal,
                                 q.shape[3] ** -0.5, docs=docs)


FIXED_DOCS = [0, 1, 2, 130, 255, 256, 900, 901, 1024]


@pytest.mark.parametrize("kind,P", [("contiguous", 4), ("zigzag", 2), ("striped", 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_layouts_with_documents(kind, P, causal):
    q, k, v = _qkv(21, 1, 4, 2, 1024, 128)
    ref = _ref(q, k, v, causal, FIXED_DOCS)
    O, m, l = layout_run(q.to(DEV), k.to(DEV), v.to(DEV), P, kind, causal,
                         out_dtype=torch.float32, docs=FIXED_DOCS)
    device_status()
    assert_bf16(O, m, l, *ref, what=f"{kind} causal={causal}")


@pytest.mark.parametrize("D", [64, 96])
def test_bf16_documents_other_head_dims(D):
    q, k, v = _qkv(22, 2, 2, 1, 640, D)
    docs = workloads.packed_documents(640, 3, 60)
    ref = _ref(q, k, v, True, docs)
    kc = [t.contiguous().to(DEV) for t in torch.split(k, [300, 340], dim=2)]
    vc = [t.contiguous().to(DEV) for t in torch.split(v, [300, 340], dim=2)]
    O, m, l = ring_attention(q.to(DEV), kc, vc, causal=True, docs=docs)
    device_status()
    assert_bf16(O, m, l, *ref)


def test_bf16_queries_whose_document_has_no_keys():
    """Keys cover documents 0 and 1 only: the rows of document 2 get O = 0,
    l = 0, m = -inf; a ragged query count and one-key chunks on the side."""
    q, k, v = _qkv(23, 1, 2, 2, 333, 128)
    docs = [0, 100, 200, 333]
    kk, vv = k[:, :, :200], v[:, :, :200]
    ref = oracle.full_attention(f64(q), f64(kk), f64(vv), np.arange(333), np.arange(200), False,
                                128 ** -0.5, docs=docs)
    lens = [1, 99, 100]
    kc = [t.contiguous().to(DEV) for t in torch.split(kk, lens, dim=2)]
    vc = [t.contiguous().to(DEV) for t in torch.split(vv, lens, dim=2)]
    O, m, l = ring_attention(q.to(DEV), kc, vc, docs=docs, out_dtype=torch.float32)
    device_status()
    assert_bf16(O, m, l, *ref)
    assert float(O[:, :, 200:].abs().max()) == 0.0
    assert torch.isneginf(m[:, :, 200:]).all() and float(l[:, :, 200:].abs().max()) == 0.0


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_8k_packed_split_units(causal):
    """The 8K workload's shape (8 heads, head_dim 128) packed with ~40
    documents; 256 work units over the grid, so units are split between CTAs
    (the stream-K tail). Sampled rows of two heads against the oracle."""
    S = 8192
    q, k, v = _qkv(24, 1, 8, 8, S, 128)
    docs = workloads.packed_documents(S, 5, 256)
    kc = [t.contiguous().to(DEV) for t in torch.split(k, 1024, dim=2)]
    vc = [t.contiguous().to(DEV) for t in torch.split(v, 1024, dim=2)]
    O, m, l = ring_attention(q.to(DEV), kc, vc, causal=causal, docs=docs, out_dtype=torch.float32)
    device_status()
    rows = sample_rows(S, docs[1:-1], 48, seed=9)
    heads = [0, 5]
    Or, Mr, Lr = oracle_rows(q, k, v, causal, 128 ** -0.5, heads, rows, docs=docs)
    got = [t[0][heads][:, rows] for t in (O, m, l)]
    assert_bf16(*got, Or, Mr, Lr)


def test_fp32_path_with_documents():
    q, k, v = _qkv(25, 1, 2, 1, 256, 64, torch.float32)
    docs = workloads.packed_documents(256, 4, 20)
    for causal in (False, True):
        ref = _ref(q, k, v, causal, docs)
        O, m, l = layout_run(q.to(DEV), k.to(DEV), v.to(DEV), 4, "zigzag", causal, docs=docs)
        device_status()
        assert_f32(O, m, l, *ref)


def test_chunk_stats_with_documents():
    q, k, v = _qkv(26, 1, 2, 2, 512, 128)
    docs = [0, 200, 330, 512]
    pos = np.arange(512)
    ref = oracle.chunk_stats(f64(q), f64(k[:, :, 128:384]), f64(v[:, :, 128:384]), pos,
                             pos[128:384], True, 128 ** -0.5, docs=docs)
    u, l, m = chunk_stats(q.to(DEV), k[:, :, 128:384].contiguous().to(DEV),
                          v[:, :, 128:384].contiguous().to(DEV), spans=[(256, 128, 1)],
                          causal=True, docs=docs)
    device_status()
    u_ref, l_ref, m_ref = ref
    O_ref = oracle.normalize(u_ref, l_ref)
    O = torch.where(l.unsqueeze(-1) > 0, u / l.clamp_min(1e-30).unsqueeze(-1), torch.zeros_like(u))
    assert_bf16(O, m, l, O_ref, m_ref, l_ref)


def test_host_entry_with_documents():
    q, k, v = _qkv(27, 1, 4, 4, 768, 128)
    docs = workloads.packed_documents(768, 6, 90)
    ref = _ref(q, k, v, True, docs)
    kc = [t.contiguous().pin_memory() for t in torch.split(k, 256, dim=2)]
    vc = [t.contiguous().pin_memory() for t in torch.split(v, 256, dim=2)]
    O, m, l = ring_attention_host(q.contiguous().pin_memory(), kc, vc, causal=True, docs=docs,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    device_status()
    assert_bf16(O, m, l, *ref)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_with_documents(causal):
    S = 896
    q, k, v = _qkv(28, 1, 4, 2, S, 128)
    g = torch.Generator(device="cpu").manual_seed(29)
    do = torch.randn(1, 4, S, 128, generator=g).to(torch.bfloat16)
    docs = [0, 1, 129, 300, 301, 640, 896]
    P, kind = 4, "zigzag"
    rs = layouts.rank_spans(kind, S, P)
    kc = [t.contiguous().to(DEV) for t in layouts.shard(k, kind, P)]
    vc = [t.contiguous().to(DEV) for t in layouts.shard(v, kind, P)]
    qs = torch.cat(layouts.shard(q, kind, P), dim=2).contiguous().to(DEV)
    dos = torch.cat(layouts.shard(do, kind, P), dim=2).contiguous().to(DEV)
    segs = [(S // P, s) for s in rs]
    O, m, l = ring_attention(qs, kc, vc, chunk_spans=rs, q_segments=segs, causal=causal, docs=docs)
    dq, dk, dv = ring_attention_bwd(qs, kc, vc, O, dos, m, l, chunk_spans=rs, q_segments=segs,
                                    causal=causal, docs=docs)
    device_status()
    dq = layouts.to_global(dq.cpu(), kind, P)
    order = np.concatenate([np.asarray(r) for r in oracle.layouts.LAYOUTS[kind](S, P)])
    inv = np.argsort(order)
    dk = torch.cat([t.cpu() for t in dk], dim=2)[:, :, inv]
    dv = torch.cat([t.cpu() for t in dv], dim=2)[:, :, inv]
    pos = np.arange(S)
    rq, rk, rv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), pos, pos, causal,
                                           128 ** -0.5, docs=docs)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        got = f64(got)
        assert not np.isnan(got).any(), name
        err = np.abs(got - ref).max()
        assert err <= 1e-2 * max(np.abs(ref).max(), 1e-6), f"{name}: {err:.3e}"
    # the key of the one-position document 0 is seen by its own query only
    assert np.allclose(f64(dk)[:, :, 0], rk[:, :, 0], atol=1e-2 * np.abs(rk).max())
