"""Pins of the backward oracle (oracle.backward), on the CPU.

The oracle follows the chain rule through O = softmax(scale Q K^T) V
("Ring Attention: Distributed Reads with Online Softmax", section "Backward
must aggregate shared dependencies": gradients per key/value shard, the same
scaling and masks, checked against a single-device reference). It is pinned
here to things other than itself: torch autograd in fp64 (a library routine),
central finite differences of the oracle's own forward, closed forms, the
chunk-by-chunk aggregation the blog describes, and planted mistakes that must
fail.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import layouts as olay


def _rand(seed, B, Hq, Hkv, Sq, Sk, D):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, Sq, D))
    k = rng.standard_normal((B, Hkv, Sk, D))
    v = rng.standard_normal((B, Hkv, Sk, D))
    do = rng.standard_normal((B, Hq, Sq, D))
    return q, k, v, do


def _torch_grads(q, k, v, do, q_pos, k_pos, causal, scale):
    """fp64 autograd through an explicit masked softmax (no fused kernels)."""
    Hq, Hkv = q.shape[1], k.shape[1]
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(Hq // Hkv, dim=1)
    vv = tv.repeat_interleave(Hq // Hkv, dim=1)
    s = scale * tq @ kk.transpose(-1, -2)
    if causal:
        vis = torch.tensor(np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None])
        s = s.masked_fill(~vis, float("-inf"))
    p = torch.softmax(s, dim=-1)
    p = torch.nan_to_num(p, nan=0.0)          # rows with no visible key
    o = p @ vv
    (o * torch.tensor(do)).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal", [
    (1, 1, 1, 7, 7, 8, False),
    (2, 4, 2, 13, 13, 8, True),
    (1, 3, 1, 5, 11, 4, False),
    (1, 2, 2, 9, 9, 16, True),
])
def test_backward_matches_autograd(B, Hq, Hkv, Sq, Sk, D, causal):
    q, k, v, do = _rand(1, B, Hq, Hkv, Sq, Sk, D)
    q_pos, k_pos = np.arange(Sk - Sq, Sk), np.arange(Sk)
    scale = D ** -0.5
    dq, dk, dv = oracle.attention_backward(q, k, v, do, q_pos, k_pos, causal, scale)
    tq, tk, tv = _torch_grads(q, k, v, do, q_pos, k_pos, causal, scale)
    for a, b in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max())


def test_backward_matches_finite_differences():
    """Central differences of L = sum(dO * O) through the oracle's forward."""
    q, k, v, do = _rand(2, 1, 1, 1, 4, 5, 3)
    q_pos, k_pos, scale = np.arange(1, 5), np.arange(5), 0.7
    dq, dk, dv = oracle.attention_backward(q, k, v, do, q_pos, k_pos, True, scale)

    def loss(q_, k_, v_):
        O, _, _ = oracle.full_attention(q_, k_, v_, q_pos, k_pos, True, scale)
        return float((O * do).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if n == name else y for n, y in (("q", q), ("k", k), ("v", v))]
            args_m = [xm if n == name else y for n, y in (("q", q), ("k", k), ("v", v))]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-7, (name, idx, fd, g[idx])


def test_closed_forms():
    # identical keys: the softmax does not depend on q, so dQ = 0; dV splits dO evenly
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 2, 6, 4))
    k = np.repeat(rng.standard_normal((1, 1, 1, 4)), 5, axis=2)
    v = rng.standard_normal((1, 1, 5, 4))
    do = rng.standard_normal((1, 2, 6, 4))
    pos_q, pos_k = np.arange(6), np.arange(5)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, pos_q, pos_k, False, 0.5)
    assert np.abs(dq).max() <= 1e-14
    assert np.allclose(dv[0, 0], np.repeat(do[0].sum(axis=(0, 1))[None, :] / 5, 5, axis=0), atol=1e-13)
    # one key: P = 1, so dS = 0, dQ = dK = 0 and dV = sum of dO over rows and heads
    k1, v1 = k[:, :, :1], v[:, :, :1]
    dq, dk, dv = oracle.attention_backward(q, k1, v1, do, pos_q, pos_k[:1], False, 0.5)
    assert np.abs(dq).max() <= 1e-14 and np.abs(dk).max() <= 1e-14
    assert np.allclose(dv[0, 0, 0], do[0].sum(axis=(0, 1)), atol=1e-13)


def test_fully_masked_rows_get_no_gradient():
    q, k, v, do = _rand(4, 1, 1, 1, 4, 4, 3)
    q_pos, k_pos = np.array([-3, -1, 0, 2]), np.arange(4)     # rows 0, 1 see no key
    dq, dk, dv = oracle.attention_backward(q, k, v, do, q_pos, k_pos, True, 1.0)
    assert np.abs(dq[0, 0, :2]).max() == 0.0
    dq2, dk2, dv2 = oracle.attention_backward(q[:, :, 2:], k, v, do[:, :, 2:], q_pos[2:], k_pos,
                                              True, 1.0)
    assert np.allclose(dk, dk2, atol=1e-14) and np.allclose(dv, dv2, atol=1e-14)


@pytest.mark.parametrize("kind,P,causal", [("contiguous", 4, True), ("zigzag", 2, True),
                                           ("striped", 4, True), ("contiguous", 3, False)])
def test_chunked_aggregation_equals_definition(kind, P, causal):
    """Per-chunk recomputation with the global statistics, gradients summed per
    chunk (the blog's aggregation) gives the definition's gradients."""
    S, D = 24, 8
    q, k, v, do = _rand(5, 1, 4, 2, S, S, D)
    pos = np.arange(S)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, pos, pos, causal, D ** -0.5)
    ranks = olay.LAYOUTS[kind](S, P)
    kc = [k[:, :, r] for r in ranks]
    vc = [v[:, :, r] for r in ranks]
    dq2, dkc, dvc = oracle.ring_attention_backward(q, kc, vc, do, pos, ranks, causal, D ** -0.5)
    assert np.abs(dq2 - dq).max() <= 1e-12
    for r, a, b in zip(ranks, dkc, dvc):
        assert np.abs(a - dk[:, :, r]).max() <= 1e-12
        assert np.abs(b - dv[:, :, r]).max() <= 1e-12


def test_chunks_of_one_key():
    S, D = 9, 4
    q, k, v, do = _rand(6, 1, 2, 1, S, S, D)
    pos = np.arange(S)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, pos, pos, True, 0.5)
    kc = [k[:, :, i:i + 1] for i in range(S)]
    vc = [v[:, :, i:i + 1] for i in range(S)]
    dq2, dkc, dvc = oracle.ring_attention_backward(q, kc, vc, do, pos, [[i] for i in range(S)],
                                                   True, 0.5)
    assert np.abs(dq2 - dq).max() <= 1e-12
    assert np.abs(np.concatenate(dkc, axis=2) - dk).max() <= 1e-12
    assert np.abs(np.concatenate(dvc, axis=2) - dv).max() <= 1e-12


def _planted(kind):
    """Copies of the definition with one plausible mistake each."""
    def f(q, k, v, do, q_pos, k_pos, causal, scale):
        s = np.where(oracle.attention._visible(q_pos, k_pos, causal),
                     scale * (q[0, 0] @ k[0, 0].T), -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        dp = do[0, 0] @ v[0, 0].T
        ds = p * dp if kind == "no_rowsum" else p * (dp - (p * dp).sum(axis=1, keepdims=True))
        dv = (p @ do[0, 0]) if kind == "p_not_transposed" else p.T @ do[0, 0]
        dq = (ds @ k[0, 0]) * (1.0 if kind == "no_scale" else scale)
        dk = scale * (ds.T @ q[0, 0])
        return dq[None, None], dk[None, None], dv[None, None]
    return f


@pytest.mark.parametrize("kind", ["no_rowsum", "no_scale", "p_not_transposed"])
def test_planted_mistakes_fail_the_autograd_pin(kind):
    q, k, v, do = _rand(7, 1, 1, 1, 6, 6, 4)
    pos = np.arange(6)
    ref = _torch_grads(q, k, v, do, pos, pos, True, 0.5)
    got = _planted(kind)(q, k, v, do, pos, pos, True, 0.5)
    assert max(np.abs(a - b).max() for a, b in zip(got, ref)) > 1e-3
    # the unplanted copy passes
    ok = oracle.attention_backward(q, k, v, do, pos, pos, True, 0.5)
    assert max(np.abs(a - b).max() for a, b in zip(ok, ref)) <= 1e-12


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def _rounded_backward(q, k, v, do, pos_q, pos_k, causal, scale, round_fn):
    """The definition with P and dS passed through ``round_fn`` before their
    products (single head group of one head each)."""
    s = np.where(olay_vis(pos_q, pos_k, causal), scale * (q @ k.T), -np.inf)
    m = s.max(axis=1)
    w = np.exp(s - m[:, None])
    p = w / w.sum(axis=1, keepdims=True)
    dp = do @ v.T
    ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    pr, dsr = round_fn(p), round_fn(ds)
    return scale * (dsr @ k), scale * (dsr.T @ q), pr.T @ do


def olay_vis(pos_q, pos_k, causal):
    return (pos_k[None, :] <= pos_q[:, None]) if causal else np.ones((len(pos_q), len(pos_k)), bool)


@pytest.mark.parametrize("causal", [False, True])
def test_rounding_bounds_hold_for_bf16_rounded_probabilities(causal):
    """The elementwise bound of the parity tests holds for a backward that
    rounds P and dS to bf16 (unit roundoff 2^-8), and is not loose: the worst
    element uses a sizeable share of it. Coarser rounding (unit roundoff
    2^-5) breaks it."""
    rng = np.random.default_rng(21)
    Sq, Sk, D = 96, 160, 32
    q = _bf16(rng.standard_normal((Sq, D)))
    k = _bf16(rng.standard_normal((Sk, D)))
    v = _bf16(rng.standard_normal((Sk, D)))
    do = _bf16(rng.standard_normal((Sq, D)))
    pq, pk = np.arange(Sk - Sq, Sk), np.arange(Sk)
    scale = D ** -0.5
    ref = oracle.attention_backward(q[None, None], k[None, None], v[None, None], do[None, None],
                                    pq, pk, causal, scale)
    bnd = oracle.gradient_rounding_bounds(q[None, None], k[None, None], v[None, None],
                                          do[None, None], pq, pk, causal, scale)
    got = _rounded_backward(q, k, v, do, pq, pk, causal, scale, _bf16)
    worst = 0.0
    for g, r, bd in zip(got, ref, bnd):
        err = np.abs(g - r[0, 0])
        assert (err <= bd[0, 0] + 1e-12).all()
        worst = max(worst, float((err / np.maximum(bd[0, 0], 1e-300)).max()))
    assert worst > 0.05, worst

    def coarse(x):  # round to 5 significant bits: unit roundoff 2^-5
        e = np.floor(np.log2(np.where(x != 0, np.abs(x), 1.0)))
        return np.round(x / 2.0 ** (e - 4)) * 2.0 ** (e - 4)

    got = _rounded_backward(q, k, v, do, pq, pk, causal, scale, coarse)
    assert any((np.abs(g - r[0, 0]) > bd[0, 0]).any() for g, r, bd in zip(got, ref, bnd))
