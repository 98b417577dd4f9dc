"""Pins of the oracle's document (packed variable-length) masks.

The pages do not treat packed sequences; the reading implemented is that a
document is a range of global positions [b_d, b_{d+1}) and that a query sees
only the keys of its own document, with the causal rule of "Ring Attention:
Distributed Reads with Online Softmax", section "Causal masks depend on
global positions", on top. These tests tie that reading to something other
than the masked code itself: a packed problem must equal its documents
solved one at a time with no document mask (documents are independent
problems), and a few closed forms.
"""
import numpy as np
import pytest

import oracle


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _per_document(fn, q, k, v, q_pos, k_pos, causal, scale, docs):
    """Solve each document on its own (rows and keys of that document only)
    with the unmasked oracle; scatter the rows back."""
    B, Hq, Sq, D = q.shape
    O = np.zeros((B, Hq, Sq, v.shape[3]))
    m = np.full((B, Hq, Sq), -np.inf)
    l = np.zeros((B, Hq, Sq))
    for d in range(len(docs) - 1):
        qi = np.nonzero((q_pos >= docs[d]) & (q_pos < docs[d + 1]))[0]
        ki = np.nonzero((k_pos >= docs[d]) & (k_pos < docs[d + 1]))[0]
        if qi.size == 0:
            continue
        o_d, m_d, l_d = fn(q[:, :, qi], k[:, :, ki], v[:, :, ki], q_pos[qi], k_pos[ki], causal,
                           scale)
        O[:, :, qi], m[:, :, qi], l[:, :, qi] = o_d, m_d, l_d
    return O, m, l


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2)])
def test_packed_equals_documents_solved_separately(causal, Hq, Hkv):
    rng = np.random.default_rng(5)
    S, D = 61, 8
    docs = [0, 1, 17, 18, 40, 61]          # lengths 1, 16, 1, 22, 21
    q, k, v = _rand(rng, 2, Hq, S, D), _rand(rng, 2, Hkv, S, D), _rand(rng, 2, Hkv, S, D)
    pos = np.arange(S)
    got = oracle.full_attention(q, k, v, pos, pos, causal, 0.3, docs=docs)
    ref = _per_document(oracle.full_attention, q, k, v, pos, pos, causal, 0.3, docs)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_documents_with_offset_and_permuted_positions():
    """Boundaries that do not start at 0, and rows whose positions are not in
    order (a zigzag-like permutation of the queries)."""
    rng = np.random.default_rng(6)
    S, D = 48, 4
    docs = [100, 113, 130, 148]
    pos = 100 + np.arange(S)
    perm = np.concatenate([pos[:12], pos[36:], pos[12:36]])
    q, k, v = _rand(rng, 1, 2, S, D), _rand(rng, 1, 1, S, D), _rand(rng, 1, 1, S, D)
    for causal in (False, True):
        got = oracle.full_attention(q, k, v, perm, pos, causal, 0.5, docs=docs)
        ref = _per_document(oracle.full_attention, q, k, v, perm, pos, causal, 0.5, docs)
        for a, b in zip(got, ref):
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_one_document_is_no_mask():
    rng = np.random.default_rng(7)
    q, k, v = _rand(rng, 1, 2, 20, 4), _rand(rng, 1, 2, 30, 4), _rand(rng, 1, 2, 30, 4)
    qp, kp = np.arange(10, 30), np.arange(30)
    for causal in (False, True):
        a = oracle.full_attention(q, k, v, qp, kp, causal, 0.7, docs=[0, 30])
        b = oracle.full_attention(q, k, v, qp, kp, causal, 0.7)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


def test_single_position_documents_closed_form():
    """Every document holds one position: each query sees exactly its own
    key, so O = v, l = 1, m = scale * <q, k> (causal or not)."""
    rng = np.random.default_rng(8)
    S, D = 9, 5
    q, k, v = _rand(rng, 1, 1, S, D), _rand(rng, 1, 1, S, D), _rand(rng, 1, 1, S, D)
    pos = np.arange(S)
    docs = np.arange(S + 1)
    for causal in (False, True):
        O, m, l = oracle.full_attention(q, k, v, pos, pos, causal, 0.25, docs=docs)
        np.testing.assert_allclose(O, v, rtol=1e-15, atol=0)
        np.testing.assert_array_equal(l, np.ones_like(l))
        np.testing.assert_allclose(m[0, 0], 0.25 * np.einsum("sd,sd->s", q[0, 0], k[0, 0]),
                                   rtol=1e-15, atol=1e-15)


def test_query_whose_document_has_no_keys():
    """Keys only in document 0; queries of document 1 see nothing: O = 0,
    l = 0, m = -inf."""
    rng = np.random.default_rng(9)
    q, k, v = _rand(rng, 1, 1, 8, 4), _rand(rng, 1, 1, 5, 4), _rand(rng, 1, 1, 5, 4)
    O, m, l = oracle.full_attention(q, k, v, np.arange(8), np.arange(5), False, 1.0,
                                    docs=[0, 5, 8])
    assert (O[0, 0, 5:] == 0).all() and (l[0, 0, 5:] == 0).all()
    assert np.isneginf(m[0, 0, 5:]).all() and np.isfinite(m[0, 0, :5]).all()


@pytest.mark.parametrize("causal", [False, True])
def test_ring_with_documents_is_chunking_invariant(causal):
    """The chunked method with documents (stats per chunk, merges) equals the
    definition, for chunks that cut across document boundaries, down to
    one-key chunks."""
    rng = np.random.default_rng(10)
    S, D = 33, 6
    docs = [0, 7, 8, 20, 33]
    q, k, v = _rand(rng, 1, 2, S, D), _rand(rng, 1, 1, S, D), _rand(rng, 1, 1, S, D)
    pos = np.arange(S)
    ref = oracle.full_attention(q, k, v, pos, pos, causal, 0.4, docs=docs)
    for cuts in ([0, 5, 19, 33], list(range(S + 1))):
        kc = [k[:, :, a:b] for a, b in zip(cuts[:-1], cuts[1:])]
        vc = [v[:, :, a:b] for a, b in zip(cuts[:-1], cuts[1:])]
        pc = [pos[a:b] for a, b in zip(cuts[:-1], cuts[1:])]
        got = oracle.ring_attention(q, kc, vc, pos, pc, causal, 0.4, docs=docs)
        for a, b in zip(got, ref):
            np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_attention_rows_with_documents():
    rng = np.random.default_rng(11)
    S, D = 40, 4
    docs = [0, 13, 40]
    q, k, v = _rand(rng, 1, 2, S, D), _rand(rng, 1, 2, S, D), _rand(rng, 1, 2, S, D)
    pos = np.arange(S)
    rows = [(0, 0, 0), (0, 1, 12), (0, 0, 13), (0, 1, 39)]
    for causal in (False, True):
        O, m, l = oracle.full_attention(q, k, v, pos, pos, causal, 0.5, docs=docs)
        Or, mr, lr = oracle.attention_rows(q, k, v, pos, pos, causal, 0.5, rows, docs=docs)
        for j, (b, h, i) in enumerate(rows):
            np.testing.assert_allclose(Or[j], O[b, h, i], rtol=1e-13, atol=1e-14)
            assert mr[j] == pytest.approx(m[b, h, i], rel=1e-14)
            assert lr[j] == pytest.approx(l[b, h, i], rel=1e-13)


def test_unmasked_pairs_closed_form():
    """A document of n positions holds n^2 visible pairs, or n(n+1)/2 with
    the causal rule; queries and keys at all positions."""
    lens = [1, 5, 128, 7]
    docs = np.concatenate([[0], np.cumsum(lens)])
    pos = np.arange(docs[-1])
    assert oracle.unmasked_pairs(pos, pos, False, docs) == sum(n * n for n in lens)
    assert oracle.unmasked_pairs(pos, pos, True, docs) == sum(n * (n + 1) // 2 for n in lens)
    # against the boolean mask on a shuffled subset
    rng = np.random.default_rng(12)
    qp = rng.choice(pos, 60, replace=False)
    kp = rng.choice(pos, 90, replace=False)
    for causal in (False, True):
        assert oracle.unmasked_pairs(qp, kp, causal, docs) == int(
            oracle.attention._visible(qp, kp, causal, docs).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_packed_equals_documents_solved_separately(causal):
    rng = np.random.default_rng(13)
    S, D = 30, 4
    docs = [0, 11, 12, 30]
    q, k, v = _rand(rng, 1, 4, S, D), _rand(rng, 1, 2, S, D), _rand(rng, 1, 2, S, D)
    do = _rand(rng, 1, 4, S, D)
    pos = np.arange(S)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, pos, pos, causal, 0.6, docs=docs)
    for d in range(len(docs) - 1):
        sl = slice(docs[d], docs[d + 1])
        rq, rk, rv = oracle.attention_backward(q[:, :, sl], k[:, :, sl], v[:, :, sl],
                                               do[:, :, sl], pos[sl], pos[sl], causal, 0.6)
        np.testing.assert_allclose(dq[:, :, sl], rq, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk[:, :, sl], rk, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv[:, :, sl], rv, rtol=0, atol=1e-12)
    # the chunked form (forward statistics, per-chunk gradients) agrees
    cuts = [0, 9, 21, 30]
    kc = [k[:, :, a:b] for a, b in zip(cuts[:-1], cuts[1:])]
    vc = [v[:, :, a:b] for a, b in zip(cuts[:-1], cuts[1:])]
    pc = [pos[a:b] for a, b in zip(cuts[:-1], cuts[1:])]
    cq, ck, cv = oracle.ring_attention_backward(q, kc, vc, do, pos, pc, causal, 0.6, docs=docs)
    np.testing.assert_allclose(cq, dq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(ck, axis=2), dk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(cv, axis=2), dv, rtol=0, atol=1e-12)


def test_bad_boundaries_rejected():
    with pytest.raises(ValueError):
        oracle.document_of([0, 1], [0, 0, 4])
    with pytest.raises(ValueError):
        oracle.document_of([5], [0, 4])
    with pytest.raises(ValueError):
        oracle.document_of([0], [3, 9])


def test_planted_boundary_slip_is_caught(monkeypatch):
    """A document lookup that puts each boundary position into the previous
    document (an off-by-one at b_d) must fail the per-document pin."""
    import oracle.attention as A

    def bad_document_of(pos, docs):
        b = np.asarray(docs, dtype=np.int64)
        return np.clip(np.searchsorted(b, np.asarray(pos), side="left") - 1, 0, b.size - 2)
    monkeypatch.setattr(A, "document_of", bad_document_of)
    with pytest.raises(AssertionError):
        test_packed_equals_documents_solved_separately(True, 2, 2)
