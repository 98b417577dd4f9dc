"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small and medium cases: the oracle evaluates every row. Sizes span several
128-row tiles and ragged tails; chunk lengths include 1, 127 and 129.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from blockwise_attention_online_gb300 import (chunk_stats, device_status, layouts, merge_lse,
                                              merge_stats, ring_attention, stats_to_lse,
                                              workloads)
from _util import (assert_bf16, assert_f32, f64, layout_run)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _full_ref(q, k, v, causal, scale, qpos=None, kpos=None):
    S = k.shape[2]
    qpos = np.arange(q.shape[2]) if qpos is None else qpos
    kpos = np.arange(S) if kpos is None else kpos
    return oracle.full_attention(f64(q), f64(k), f64(v), qpos, kpos, causal, scale)


def _split(t, lens):
    return [x.contiguous() for x in torch.split(t, lens, dim=2)]


# ------------------------------------------------------------------ fp32

@pytest.fixture(scope="module")
def cfg1():
    w = workloads.WORKLOADS["fp32_256"]
    q, k, v = workloads.make_qkv(w)          # CPU generator, seed 0
    return w, q, k, v


def test_fp32_cfg1_four_chunks_ring(cfg1):
    """fp32, 256 x 256, head_dim 64, 4 contiguous chunks of 64, ring order."""
    w, q, k, v = cfg1
    ref = _full_ref(q, k, v, False, w.scale)
    O, m, l = layout_run(q.to(DEV), k.to(DEV), v.to(DEV), 4, "contiguous", False)
    device_status()
    assert_f32(O, m, l, *ref)


def test_fp32_cfg1_size1_chunks(cfg1):
    """The same problem re-run with 256 chunks of one key each."""
    w, q, k, v = cfg1
    ref = _full_ref(q, k, v, False, w.scale)
    kc = _split(k.to(DEV), [1] * 256)
    vc = _split(v.to(DEV), [1] * 256)
    O, m, l = ring_attention(q.to(DEV), kc, vc)
    device_status()
    assert_f32(O, m, l, *ref)


@pytest.mark.parametrize("kind", ["contiguous", "zigzag", "striped"])
def test_fp32_cfg1_causal_layouts(cfg1, kind):
    w, q, k, v = cfg1
    ref = _full_ref(q, k, v, True, w.scale)
    O, m, l = layout_run(q.to(DEV), k.to(DEV), v.to(DEV), 4, kind, True)
    device_status()
    assert_f32(O, m, l, *ref)


def test_fp32_scalar_two_shards():
    """Blog, "Do not average independently normalized shard outputs": shard A
    (score 0, value 0), shard B (score 10, value 1) -> e^10 / (1 + e^10)."""
    q, ks, vs = workloads.scalar_two_shards()
    q = q.to(DEV)
    sa = chunk_stats(q, ks[0].to(DEV), vs[0].to(DEV), scale=1.0)
    sb = chunk_stats(q, ks[1].to(DEV), vs[1].to(DEV), scale=1.0, spans=[(1, 1, 1)])
    assert sa[0].item() == 0.0 and sa[1].item() == 1.0 and sa[2].item() == 0.0
    assert sb[0].item() == 1.0 and sb[1].item() == 1.0 and sb[2].item() == 10.0
    u, l, m = merge_stats(*[t.clone() for t in sa], *sb)
    o = (u / l.unsqueeze(-1)).item()
    assert abs(o - math.exp(10) / (1 + math.exp(10))) < 1e-6
    assert m.item() == 10.0
    O, M, L = ring_attention(q, [k.to(DEV) for k in ks], [v.to(DEV) for v in vs], scale=1.0)
    assert abs(O.item() - math.exp(10) / (1 + math.exp(10))) < 1e-6
    assert M.item() == 10.0 and abs(L.item() - (1 + math.exp(-10))) < 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_fp32_stats_then_merge_chain(cfg1, causal):
    """chunk_stats per chunk + merge_stats chain == ordinary attention."""
    w, q, k, v = cfg1
    ref = _full_ref(q, k, v, causal, w.scale)
    lens = [1, 63, 128, 64]
    qd = q.to(DEV)
    acc = None
    start = 0
    for kc, vc in zip(_split(k.to(DEV), lens), _split(v.to(DEV), lens)):
        st = chunk_stats(qd, kc, vc, spans=[(kc.shape[2], start, 1)], causal=causal)
        start += kc.shape[2]
        acc = [t.clone() for t in st] if acc is None else merge_stats(*acc, *st)
    u, l, m = acc
    O = torch.where(l.unsqueeze(-1) > 0, u / l.unsqueeze(-1), torch.zeros_like(u))
    device_status()
    assert_f32(O, m, l, *ref)


def test_fp32_chunk_stats_match_oracle(cfg1):
    w, q, k, v = cfg1
    pos = np.arange(256)
    u_ref, l_ref, m_ref = oracle.chunk_stats(f64(q), f64(k[:, :, 64:192]), f64(v[:, :, 64:192]),
                                             pos, pos[64:192], True, w.scale)
    u, l, m = chunk_stats(q.to(DEV), k[:, :, 64:192].contiguous().to(DEV),
                          v[:, :, 64:192].contiguous().to(DEV), spans=[(128, 64, 1)], causal=True)
    device_status()
    fin = np.isfinite(m_ref)
    assert np.array_equal(np.isfinite(f64(m)), fin)
    assert np.abs(f64(m)[fin] - m_ref[fin]).max() <= 1e-5
    assert np.abs(f64(u) - u_ref).max() <= 1e-5 * max(1.0, l_ref.max())
    assert (np.abs(f64(l) - l_ref) <= 1e-5 * np.maximum(1, l_ref)).all()


def test_merge_kernel_edge_cases():
    """-inf sides, both -inf, and a head_dim that is not a multiple of 4."""
    g = torch.Generator(device="cpu").manual_seed(3)
    for D in (5, 64):
        rows = 37
        u1 = torch.randn(rows, D, generator=g); u2 = torch.randn(rows, D, generator=g)
        l1 = torch.rand(rows, generator=g) + 0.5; l2 = torch.rand(rows, generator=g) + 0.5
        m1 = torch.randn(rows, generator=g) * 5; m2 = torch.randn(rows, generator=g) * 5
        m1[3] = -math.inf; u1[3] = 0; l1[3] = 0
        m2[4] = -math.inf; u2[4] = 0; l2[4] = 0
        m1[5] = m2[5] = -math.inf; u1[5] = u2[5] = 0; l1[5] = l2[5] = 0
        ref = oracle.merge_stats((f64(u1), f64(l1), f64(m1)), (f64(u2), f64(l2), f64(m2)))
        acc = [t.to(DEV) for t in (u1, l1, m1)]
        merge_stats(*acc, *[t.to(DEV) for t in (u2, l2, m2)])
        device_status()
        assert np.abs(f64(acc[0]) - ref[0]).max() <= 1e-5 * np.abs(ref[0]).max()
        assert np.allclose(f64(acc[1]), ref[1], rtol=1e-6, atol=0)
        assert np.array_equal(f64(acc[2]), ref[2].astype(np.float32).astype(np.float64))


# ------------------------------------------------------------------ bf16

def _bf16_inputs(B, Hq, Hkv, S, D, seed, Sq=None):
    g = torch.Generator(device="cpu").manual_seed(seed)
    Sq = S if Sq is None else Sq
    q = torch.randn(B, Hq, Sq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("D", [64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,lens", [(1, [1]), (128, [128]), (300, [1, 127, 129, 43]),
                                    (520, [520]), (700, [256, 200, 244])])
def test_bf16_small_ragged(D, causal, S, lens):
    q, k, v = _bf16_inputs(1, 2, 1, S, D, seed=S + D + causal)
    ref = _full_ref(q, k, v, causal, 1 / math.sqrt(D))
    kc = _split(k.to(DEV), lens)
    vc = _split(v.to(DEV), lens)
    O, m, l = ring_attention(q.to(DEV), kc, vc, causal=causal)
    device_status()
    assert_bf16(O, m, l, *ref, what=f"S={S} D={D} causal={causal}")


@pytest.mark.parametrize("kind", ["contiguous", "zigzag", "striped"])
def test_bf16_layouts_gqa(kind):
    """GQA 4:1, 4 virtual ranks, each layout; rows compared in global order."""
    q, k, v = _bf16_inputs(2, 8, 2, 1024, 128, seed=17)
    ref = _full_ref(q, k, v, True, 1 / math.sqrt(128))
    O, m, l = layout_run(q.to(DEV), k.to(DEV), v.to(DEV), 4, kind, True)
    device_status()
    assert_bf16(O, m, l, *ref, what=kind)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_chunk_stats_then_merge(causal):
    q, k, v = _bf16_inputs(1, 2, 2, 640, 128, seed=5)
    ref = _full_ref(q, k, v, causal, 1 / math.sqrt(128))
    lens = [129, 255, 256]
    acc = None
    start = 0
    qd = q.to(DEV)
    for kc, vc in zip(_split(k.to(DEV), lens), _split(v.to(DEV), lens)):
        st = chunk_stats(qd, kc, vc, spans=[(kc.shape[2], start, 1)], causal=causal)
        # the chunk's own statistics against the oracle's
        pos = np.arange(640)
        u_r, l_r, m_r = oracle.chunk_stats(f64(q), f64(kc), f64(vc), pos,
                                           pos[start:start + kc.shape[2]], causal, 1 / math.sqrt(128))
        uu = f64(st[0])
        assert (np.abs(uu - u_r) <= 1e-2 * np.maximum(1.0, l_r)[..., None]).all()
        start += kc.shape[2]
        acc = [t.clone() for t in st] if acc is None else merge_stats(*acc, *st)
    u, l, m = acc
    O = torch.where(l.unsqueeze(-1) > 0, u / l.unsqueeze(-1), torch.zeros_like(u))
    device_status()
    assert_bf16(O, m, l, *ref, what="stats+merge")


def test_bf16_fully_masked_rows():
    """Queries placed before every key: O = 0, l = 0, m = -inf."""
    q, k, v = _bf16_inputs(1, 1, 1, 200, 64, seed=9, Sq=130)
    qd = q.to(DEV)
    O, m, l = ring_attention(qd, [k.to(DEV)], [v.to(DEV)], chunk_spans=[[(200, 1000, 1)]],
                             causal=True)
    device_status()
    assert torch.all(O == 0) and torch.all(l == 0) and torch.all(torch.isneginf(m))


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_fp32_output_matches_bf16_output(causal):
    """The fp32-O option changes only the final store: the bf16 O is the fp32
    O rounded to nearest even, and m, l are identical."""
    q, k, v = _bf16_inputs(1, 2, 2, 700, 128, seed=23)
    kc = _split(k.to(DEV), [300, 400]); vc = _split(v.to(DEV), [300, 400])
    O32, m32, l32 = ring_attention(q.to(DEV), kc, vc, causal=causal, out_dtype=torch.float32)
    O16, m16, l16 = ring_attention(q.to(DEV), kc, vc, causal=causal)
    device_status()
    assert O32.dtype == torch.float32 and O16.dtype == torch.bfloat16
    assert torch.equal(O32.to(torch.bfloat16), O16)
    assert torch.equal(m32, m16) and torch.equal(l32, l16)
    ref = _full_ref(q, k, v, causal, 1 / math.sqrt(128))
    assert_bf16(O32, m32, l32, *ref, what="fp32 O")


def test_bf16_cfg2_full_oracle():
    """bf16, 8 heads, 8192 x 8192, head_dim 128, 8 contiguous chunks of 1024 in
    ring order over 8 query segments; every row checked."""
    w = workloads.WORKLOADS["bf16_8k"]
    q, k, v = workloads.make_qkv(w)
    ref = _full_ref(q, k, v, False, w.scale)
    O, m, l = layout_run(q.to(DEV), k.to(DEV), v.to(DEV), 8, "contiguous", False)
    device_status()
    assert_bf16(O, m, l, *ref, what="cfg2")
    # bitwise repeatable
    O2, m2, l2 = layout_run(q.to(DEV), k.to(DEV), v.to(DEV), 8, "contiguous", False)
    assert torch.equal(O, O2) and torch.equal(m, m2) and torch.equal(l, l2)


@pytest.mark.parametrize("kind", ["zigzag", "striped"])
def test_bf16_head_dim_96_layouts(kind):
    """head_dim 96 (a non-power-of-two width; the second 64-column box of every
    tile is half zero fill): GQA 4:1 over 4 virtual ranks, causal."""
    q, k, v = _bf16_inputs(1, 8, 2, 1024, 96, seed=19)
    ref = _full_ref(q, k, v, True, 1 / math.sqrt(96))
    O, m, l = layout_run(q.to(DEV), k.to(DEV), v.to(DEV), 4, kind, True)
    device_status()
    assert_bf16(O, m, l, *ref, what=f"D=96 {kind}")


@pytest.mark.parametrize("out_dtype", [None, torch.float32])
def test_bf16_head_dim_96_split_units(out_dtype):
    """Enough units that the last rounds are split across CTAs (partial results
    published and merged), head_dim 96, bf16 and fp32 O."""
    q, k, v = _bf16_inputs(1, 4, 4, 2304, 96, seed=23)
    ref = _full_ref(q, k, v, False, 1 / math.sqrt(96))
    kc = _split(k.to(DEV), [1024, 1280])
    vc = _split(v.to(DEV), [1024, 1280])
    O, m, l = ring_attention(q.to(DEV), kc, vc, causal=False, out_dtype=out_dtype)
    device_status()
    assert_bf16(O, m, l, *ref, what="D=96 split")


def test_bf16_head_dim_96_chunk_stats():
    q, k, v = _bf16_inputs(1, 2, 1, 384, 96, seed=29)
    pos = np.arange(384)
    u, l, m = chunk_stats(q.to(DEV), k[:, :, 128:].contiguous().to(DEV),
                          v[:, :, 128:].contiguous().to(DEV), spans=[(256, 128, 1)], causal=True)
    device_status()
    u_r, l_r, m_r = oracle.chunk_stats(f64(q), f64(k[:, :, 128:]), f64(v[:, :, 128:]), pos,
                                       pos[128:], True, 1 / math.sqrt(96))
    fin = np.isfinite(m_r)
    assert np.array_equal(np.isfinite(f64(m)), fin)
    assert (np.abs(f64(u) - u_r) <= 1e-2 * np.maximum(1.0, l_r)[..., None]).all()
    assert (np.abs(f64(l) - l_r) <= 1e-3 * np.maximum(1.0, l_r)).all()


@pytest.mark.parametrize("D", [5, 128])
def test_merge_lse_matches_oracle(D):
    rng = np.random.default_rng(D)
    rows = 1000
    oa = rng.standard_normal((rows, D)).astype(np.float32)
    ob = rng.standard_normal((rows, D)).astype(np.float32)
    la = rng.normal(0, 6, rows).astype(np.float32)
    lb = rng.normal(0, 6, rows).astype(np.float32)
    la[:7] = -np.inf                      # empty accumulator rows
    lb[3:10] = -np.inf                    # empty new rows (3..6 empty on both sides)
    ref_o, ref_l = oracle.merge_lse((oa, la), (ob, lb))
    o_acc, l_acc = torch.tensor(oa, device=DEV), torch.tensor(la, device=DEV)
    merge_lse(o_acc, l_acc, torch.tensor(ob, device=DEV), torch.tensor(lb, device=DEV))
    device_status()
    got_l = f64(l_acc)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(got_l), fin)
    assert np.abs(got_l[fin] - ref_l[fin]).max() <= 1e-5 * max(1.0, np.abs(ref_l[fin]).max())
    assert np.abs(f64(o_acc) - ref_o).max() <= 1e-5


def test_lse_composes_ring_outputs():
    """Two groups of chunks attended separately, each (O, lse) from the ring
    kernel, merged in log-sum-exp form: equal to one call over all chunks."""
    q, k, v = _bf16_inputs(1, 4, 2, 1024, 128, seed=31)
    qd = q.to(DEV)
    kc = _split(k.to(DEV), [256, 256, 512])
    vc = _split(v.to(DEV), [256, 256, 512])
    spans = [[(256, 0, 1)], [(256, 256, 1)], [(512, 512, 1)]]
    O1, m1, l1 = ring_attention(qd, kc[:2], vc[:2], chunk_spans=spans[:2], causal=True,
                                out_dtype=torch.float32)
    O2, m2, l2 = ring_attention(qd, kc[2:], vc[2:], chunk_spans=spans[2:], causal=True,
                                out_dtype=torch.float32)
    lse1, lse2 = stats_to_lse(m1, l1), stats_to_lse(m2, l2)
    merge_lse(O1, lse1, O2, lse2)
    device_status()
    ref = _full_ref(q, k, v, True, 1 / math.sqrt(128))
    assert np.abs(f64(O1) - ref[0]).max() <= 1e-2
    lse_ref = oracle.stats_to_lse(ref[1], ref[2])
    assert np.abs(f64(lse1) - lse_ref).max() <= 1e-3 * max(1.0, np.abs(lse_ref).max())
