"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

None of these checks compares the oracle with itself: each one is a worked
example printed on a page, a closed form, a brute-force evaluation written
independently with Python scalars, a library routine the definition reduces
to, or an invariant the pages state. Planted-mistake tests at the end show
that plausible slips in the oracle make some pin fail.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import layouts as olay
from blockwise_attention_online_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.to(torch.float64).numpy()


def _split(x, sizes, axis=2):
    idx = np.cumsum(sizes)[:-1]
    return np.split(x, idx, axis=axis)


# --- worked example printed on the blog ----------------------------------

def test_scalar_example_printed_values():
    """"Ring Attention: Distributed Reads with Online Softmax", section "Do
    not average independently normalized shard outputs": averaging the two
    shards' local outputs gives 0.5, the global softmax gives about 0.99995."""
    with open(os.path.join(GOLDEN, "scalar_two_shards.json")) as f:
        gold = json.load(f)
    q, ks, vs = workloads.scalar_two_shards()
    q, ks, vs = _np(q), [_np(k) for k in ks], [_np(v) for v in vs]
    pos0 = np.array([0])
    sa = oracle.chunk_stats(q, ks[0], vs[0], pos0, pos0, False, 1.0)
    sb = oracle.chunk_stats(q, ks[1], vs[1], pos0, pos0, False, 1.0)
    # each shard alone: u = exp(0) * value, l = 1, m = its own score
    assert sa[0].item() == 0.0 and sa[1].item() == 1.0 and sa[2].item() == 0.0
    assert sb[0].item() == 1.0 and sb[1].item() == 1.0 and sb[2].item() == 10.0
    u, l, m = oracle.merge_stats(sa, sb)
    o = oracle.normalize(u, l).item()
    assert m.item() == 10.0
    assert l.item() == pytest.approx(1.0 + math.exp(-10.0), rel=1e-15)
    assert o == pytest.approx(math.exp(10) / (1 + math.exp(10)), rel=1e-15)
    digits = gold["printed"]["global_softmax_output_digits"]
    assert round(o, digits) == gold["printed"]["global_softmax_output"]
    naive = 0.5 * (oracle.normalize(*sa[:2]).item() + oracle.normalize(*sb[:2]).item())
    assert naive == gold["printed"]["average_of_local_outputs"]
    assert abs(naive - o) > 0.49
    # the ring over both shards, in both orders, gives the same
    for order in ([0, 1], [1, 0]):
        O, M, L = oracle.ring_attention(q, ks, vs, pos0, [pos0, pos0], False, 1.0, order)
        assert O.item() == pytest.approx(o, rel=1e-15) and M.item() == 10.0


def test_numerator_alone_is_insufficient():
    """"Try it" on the same blog: numerators relative to different maxima can
    not be added; with the scalar shards, adding u's and l's without the
    exp(own_max - new_max) factors gives the naive 0.5, not 0.99995."""
    q, ks, vs = (workloads.scalar_two_shards())
    q, ks, vs = _np(q), [_np(k) for k in ks], [_np(v) for v in vs]
    pos0 = np.array([0])
    sa = oracle.chunk_stats(q, ks[0], vs[0], pos0, pos0, False, 1.0)
    sb = oracle.chunk_stats(q, ks[1], vs[1], pos0, pos0, False, 1.0)
    wrong = (sa[0] + sb[0]) / (sa[1] + sb[1])[..., None]
    right = oracle.normalize(*oracle.merge_stats(sa, sb)[:2])
    assert wrong.item() == 0.5
    assert right.item() > 0.9999


# --- invariance the exercise states ---------------------------------------

@pytest.fixture(scope="module")
def cfg1():
    w = workloads.WORKLOADS["fp32_256"]
    q, k, v = workloads.make_qkv(w)
    return w, _np(q), _np(k), _np(v)


def _ring_vs_full(q, k, v, sizes, causal, scale, order=None, qpos=None, kpos=None):
    S = k.shape[2]
    kpos = np.arange(S) if kpos is None else kpos
    qpos = np.arange(q.shape[2]) if qpos is None else qpos
    O, M, L = oracle.full_attention(q, k, v, qpos, kpos, causal, scale)
    kc, vc, pc = _split(k, sizes), _split(v, sizes), _split(kpos, sizes, axis=0)
    O2, M2, L2 = oracle.ring_attention(q, kc, vc, qpos, pc, causal, scale, order)
    return (O, M, L), (O2, M2, L2)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("split", ["one", "4x64", "256x1", "random"])
def test_chunk_invariance(cfg1, split, causal):
    """Exercise task statement: ring_attention equals ordinary attention over
    the concatenated sequence for any split, even chunks of size 1."""
    w, q, k, v = cfg1
    rng = np.random.default_rng(7)
    sizes = {"one": [256], "4x64": [64] * 4, "256x1": [1] * 256,
             "random": None}[split]
    if sizes is None:
        cuts = np.sort(rng.choice(np.arange(1, 256), size=9, replace=False))
        sizes = np.diff(np.concatenate([[0], cuts, [256]])).tolist()
    (O, M, L), (O2, M2, L2) = _ring_vs_full(q, k, v, sizes, causal, w.scale)
    np.testing.assert_allclose(O2, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(M2, M, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L2, L, rtol=1e-12, atol=0)


def test_ring_visit_order_invariance(cfg1):
    """Each device walks the chunks in its own ring order (blog, "Partition
    the sequence across devices"); the result does not depend on the order."""
    w, q, k, v = cfg1
    P = 4
    assert oracle.ring_order(2, 4) == [2, 1, 0, 3]
    ref = None
    for r in range(P):
        _, (O2, M2, L2) = _ring_vs_full(q, k, v, [64] * 4, True, w.scale,
                                        order=oracle.ring_order(r, P))
        if ref is None:
            ref = (O2, M2, L2)
        for a, b in zip(ref, (O2, M2, L2)):
            np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_merge_equals_stats_of_union(cfg1):
    """Merge rule (exercise hint 2): merge(stats(A), stats(B)) == stats(A u B)
    in either order, numerator and denominator relative to the shared max."""
    w, q, k, v = cfg1
    pos = np.arange(256)
    for causal in (False, True):
        a = oracle.chunk_stats(q, k[:, :, :100], v[:, :, :100], pos, pos[:100], causal, w.scale)
        b = oracle.chunk_stats(q, k[:, :, 100:], v[:, :, 100:], pos, pos[100:], causal, w.scale)
        ab = oracle.chunk_stats(q, k, v, pos, pos, causal, w.scale)
        for merged in (oracle.merge_stats(a, b), oracle.merge_stats(b, a)):
            np.testing.assert_allclose(merged[2], ab[2], atol=0, rtol=1e-14)
            np.testing.assert_allclose(merged[1], ab[1], rtol=1e-13)
            np.testing.assert_allclose(merged[0], ab[0], rtol=1e-12, atol=1e-12)


# --- brute force with Python scalars ---------------------------------------

def _brute(q, k, v, qpos, kpos, causal, scale):
    """Softmax written out with Python floats: no max subtraction, no numpy."""
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    O = np.zeros(q.shape[:3] + (v.shape[3],))
    M = np.full(q.shape[:3], -math.inf)
    L = np.zeros(q.shape[:3])
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                sc = []
                for j in range(k.shape[2]):
                    if causal and kpos[j] > qpos[i]:
                        continue
                    s = 0.0
                    for d in range(D):
                        s += float(q[b, h, i, d]) * float(k[b, h // g, j, d])
                    sc.append((scale * s, j))
                if not sc:
                    continue
                ws = [(math.exp(s), j) for s, j in sc]
                z = sum(w for w, _ in ws)
                for w, j in ws:
                    for d in range(v.shape[3]):
                        O[b, h, i, d] += w / z * float(v[b, h // g, j, d])
                mx = max(s for s, _ in sc)
                M[b, h, i] = mx
                L[b, h, i] = z / math.exp(mx)
    return O, M, L


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 5, 3), (2, 4, 2, 7, 4), (1, 2, 1, 8, 1)])
def test_brute_force_tiny(shape, causal):
    B, Hq, Hkv, S, D = shape
    rng = np.random.default_rng(sum(shape) + causal)
    q = rng.standard_normal((B, Hq, S, D))
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    # scrambled global positions, so that local index != global position
    qpos = rng.permutation(S)
    kpos = rng.permutation(S)
    scale = 0.7
    O, M, L = oracle.full_attention(q, k, v, qpos, kpos, causal, scale)
    Ob, Mb, Lb = _brute(q, k, v, qpos, kpos, causal, scale)
    np.testing.assert_allclose(O, Ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(M, Mb, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(L, Lb, rtol=1e-12)


# --- library special case ---------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 1), (6, 3)])
def test_matches_torch_sdpa_fp64(causal, Hq, Hkv):
    """With positions equal to row indices, the definition is torch's
    scaled_dot_product_attention (fp64, CPU); grouped heads reduce to plain
    multi-head attention with each K/V head repeated for its query group."""
    g = torch.Generator().manual_seed(11 + Hq + causal)
    B, S, D = 2, 37, 16
    q = torch.randn(B, Hq, S, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, S, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, S, D, generator=g, dtype=torch.float64)
    scale = 1.0 / math.sqrt(D)
    rep = Hq // Hkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(rep, dim=1), v.repeat_interleave(rep, dim=1),
        is_causal=causal, scale=scale)
    O, _, _ = oracle.full_attention(q.numpy(), k.numpy(), v.numpy(),
                                    np.arange(S), np.arange(S), causal, scale)
    np.testing.assert_allclose(O, ref.numpy(), rtol=1e-12, atol=1e-12)


# --- closed forms ------------------------------------------------------------

def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    S, D = 9, 5
    q = rng.standard_normal((1, 1, 4, D))
    k = np.tile(rng.standard_normal((1, 1, 1, D)), (1, 1, S, 1))
    v = rng.standard_normal((1, 1, S, D))
    O, M, L = oracle.full_attention(q, k, v, np.arange(4), np.arange(S), False, 0.3)
    np.testing.assert_allclose(O[0, 0], np.broadcast_to(v[0, 0].mean(0), (4, D)), atol=1e-14)
    np.testing.assert_allclose(L, S, rtol=1e-15)
    np.testing.assert_allclose(M[0, 0], 0.3 * q[0, 0] @ k[0, 0, 0], rtol=1e-15)


def test_causal_first_row_sees_only_itself(cfg1):
    w, q, k, v = cfg1
    pos = np.arange(256)
    O, M, L = oracle.full_attention(q, k, v, pos, pos, True, w.scale)
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, 0], atol=1e-15)
    assert L[0, 0, 0] == 1.0
    assert M[0, 0, 0] == pytest.approx(w.scale * q[0, 0, 0] @ k[0, 0, 0], rel=1e-15)
    # the last row sees every key: same as the non-causal last row
    On, Mn, Ln = oracle.full_attention(q, k, v, pos, pos, False, w.scale)
    np.testing.assert_allclose(O[0, 0, -1], On[0, 0, -1], atol=1e-15)


def test_dominant_score_selects_its_value():
    rng = np.random.default_rng(5)
    S, D = 16, 4
    q = np.zeros((1, 1, 1, D)); q[..., 0] = 1.0
    k = 0.01 * rng.standard_normal((1, 1, S, D))
    k[0, 0, 11, 0] = 60.0                       # score 60 above the rest
    v = rng.standard_normal((1, 1, S, D))
    O, M, L = oracle.full_attention(q, k, v, [0], np.arange(S), False, 1.0)
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, 11], atol=1e-20 + 1e-24 * S)
    assert M.item() == 60.0
    assert L.item() == pytest.approx(1.0, abs=S * math.exp(-59))


def test_known_softmax_weights():
    """Scores 0, ln 2, ln 3 give softmax weights 1/6, 2/6, 3/6."""
    q = np.ones((1, 1, 1, 1))
    k = np.array([0.0, math.log(2), math.log(3)]).reshape(1, 1, 3, 1)
    v = np.array([6.0, 0.0, 12.0]).reshape(1, 1, 3, 1)
    O, M, L = oracle.full_attention(q, k, v, [0], [0, 1, 2], False, 1.0)
    assert O.item() == pytest.approx(1.0 + 6.0, rel=1e-15)
    assert M.item() == pytest.approx(math.log(3), rel=1e-15)
    assert L.item() == pytest.approx(6.0 / 3.0, rel=1e-15)


def test_fully_masked_rows_and_chunks():
    """A row that sees no key: u = 0, l = 0, m = -inf, output 0; merging a
    -inf side changes nothing (the masked-step rule of the IRIS ring kernel:
    a fully masked step contributes zero)."""
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 1, 3, 4))
    k = rng.standard_normal((1, 1, 5, 4))
    v = rng.standard_normal((1, 1, 5, 4))
    qpos = np.array([0, 1, 2]); kpos = np.array([3, 4, 5, 6, 7])
    u, l, m = oracle.chunk_stats(q, k, v, qpos, kpos, True, 1.0)
    assert np.all(u == 0) and np.all(l == 0) and np.all(m == -np.inf)
    O, M, L = oracle.full_attention(q, k, v, qpos, kpos, True, 1.0)
    assert np.all(O == 0) and np.all(np.isneginf(M)) and np.all(L == 0)
    other = oracle.chunk_stats(q, k, v, qpos, kpos, False, 1.0)
    for merged in (oracle.merge_stats((u, l, m), other), oracle.merge_stats(other, (u, l, m))):
        for a, b in zip(merged, other):
            np.testing.assert_array_equal(a, b)
    both = oracle.merge_stats((u, l, m), (u, l, m))
    assert not np.any(np.isnan(both[0])) and np.all(both[1] == 0)


def test_attention_rows_matches_definition(cfg1):
    w, q, k, v = cfg1
    pos = np.arange(256)
    O, M, L = oracle.full_attention(q, k, v, pos, pos, True, w.scale)
    rows = [(0, 0, i) for i in (0, 1, 63, 64, 200, 255)]
    Or, Mr, Lr = oracle.attention_rows(q, k, v, pos, pos, True, w.scale, rows)
    for n, (_, _, i) in enumerate(rows):
        np.testing.assert_allclose(Or[n], O[0, 0, i], atol=1e-13)
        assert Mr[n] == pytest.approx(M[0, 0, i], rel=1e-14)
        assert Lr[n] == pytest.approx(L[0, 0, i], rel=1e-13)


# --- layouts --------------------------------------------------------------------

def test_layout_examples():
    assert [list(x) for x in olay.contiguous(8, 2)] == [[0, 1, 2, 3], [4, 5, 6, 7]]
    # 2P = 4 blocks of 2: device 0 owns blocks 0 and 3, device 1 blocks 1 and 2
    assert [list(x) for x in olay.zigzag(8, 2)] == [[0, 1, 6, 7], [2, 3, 4, 5]]
    assert [list(x) for x in olay.striped(8, 2)] == [[0, 2, 4, 6], [1, 3, 5, 7]]
    for kind in ("contiguous", "zigzag", "striped"):
        allp = np.concatenate(olay.positions(kind, 64, 4))
        assert sorted(allp.tolist()) == list(range(64))


def test_unmasked_pairs_brute_force():
    rng = np.random.default_rng(2)
    qp, kp = rng.permutation(20), rng.permutation(13)
    n = sum(1 for a in qp for b in kp if b <= a)
    assert oracle.unmasked_pairs(qp, kp, True) == n
    assert oracle.unmasked_pairs(qp, kp, False) == 20 * 13
    # a contiguous causal sequence of n tokens has n(n+1)/2 visible pairs
    assert oracle.unmasked_pairs(np.arange(100), np.arange(100), True) == 5050


def test_zigzag_balances_causal_work():
    """Blog, "Causal masks depend on global positions": contiguous causal
    sharding is imbalanced, paired early/late chunks even it out."""
    n, P = 1024, 8
    def imbalance(kind):
        pos = olay.positions(kind, n, P)
        allk = np.arange(n)
        work = [oracle.unmasked_pairs(p, allk, True) for p in pos]
        return max(work) / (sum(work) / P)
    assert imbalance("contiguous") > 1.8
    assert imbalance("zigzag") == pytest.approx(1.0, abs=1e-12)
    assert imbalance("striped") < 1.01


# --- planted mistakes: each must make some pin fail -----------------------------

def _pins_pass(monkeypatch_target=None):
    w = workloads.WORKLOADS["fp32_256"]
    q, k, v = (_np(t) for t in workloads.make_qkv(w, S=32))
    try:
        (O, M, L), (O2, M2, L2) = _ring_vs_full(q, k, v, [8] * 4, True, w.scale)
        np.testing.assert_allclose(O2, O, atol=1e-12)
        np.testing.assert_allclose(L2, L, rtol=1e-12)
        qs, ks, vs = workloads.scalar_two_shards()
        qs, ks, vs = _np(qs), [_np(x) for x in ks], [_np(x) for x in vs]
        p = np.array([0])
        Os, _, _ = oracle.ring_attention(qs, ks, vs, p, [p, p], False, 1.0)
        assert abs(Os.item() - math.exp(10) / (1 + math.exp(10))) < 1e-12
        Ob, _, _ = _brute(q[:, :, :6], k[:, :, :6], v[:, :, :6], np.arange(6), np.arange(6), True, w.scale)
        Od, _, _ = oracle.full_attention(q[:, :, :6], k[:, :, :6], v[:, :, :6], np.arange(6), np.arange(6), True, w.scale)
        np.testing.assert_allclose(Od, Ob, atol=1e-12)
        return True
    except AssertionError:
        return False


def test_pins_pass_on_the_real_oracle():
    assert _pins_pass()


def test_planted_merge_without_rescale_is_caught(monkeypatch):
    import oracle.attention as A

    def bad_merge(acc, new):
        u1, l1, m1 = acc
        u2, l2, m2 = new
        return u1 + u2, l1 + l2, np.maximum(m1, m2)       # forgot the rescale
    monkeypatch.setattr(A, "merge_stats", bad_merge)
    assert not _pins_pass()


def test_planted_one_sided_rescale_is_caught(monkeypatch):
    import oracle.attention as A
    real = A.merge_stats

    def bad_merge(acc, new):
        u1, l1, m1 = acc
        u2, l2, m2 = new
        m = np.maximum(m1, m2)
        with np.errstate(invalid="ignore"):
            a1 = np.where(m1 == -np.inf, 0.0, np.exp(m1 - m))
        return a1[..., None] * u1 + u2, a1 * l1 + l2, m   # new side not rescaled
    monkeypatch.setattr(A, "merge_stats", bad_merge)
    assert not _pins_pass()
    assert A.merge_stats is not real


def test_planted_causal_off_by_one_is_caught(monkeypatch):
    import oracle.attention as A

    def bad_visible(q_pos, k_pos, causal, docs=None):
        q_pos = np.asarray(q_pos); k_pos = np.asarray(k_pos)
        if not causal:
            return np.ones((q_pos.size, k_pos.size), dtype=bool)
        return k_pos[None, :] < q_pos[:, None]            # excludes the diagonal
    monkeypatch.setattr(A, "_visible", bad_visible)
    assert not _pins_pass()


def test_planted_transposed_head_group_is_caught(monkeypatch):
    """GQA mapping slip (h % Hkv instead of h // group) must fail the SDPA pin."""
    import oracle.attention as A
    real = A.chunk_stats

    def bad_stats(q, k, v, q_pos, k_pos, causal, scale, docs=None):
        Hq, Hkv = q.shape[1], k.shape[1]
        idx = [h % Hkv for h in range(Hq)]
        kk = np.asarray(k)[:, idx]
        vv = np.asarray(v)[:, idx]
        return real(q, kk, vv, q_pos, k_pos, causal, scale, docs)
    monkeypatch.setattr(A, "chunk_stats", bad_stats)
    with pytest.raises(AssertionError):
        test_matches_torch_sdpa_fp64(False, 6, 3)
