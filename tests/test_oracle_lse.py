"""Pins of the log-sum-exp merge (oracle.lse): the scalar example of the blog,
equivalence with the pages' (u, l, m) merge, closed forms, and a planted
mistake that must fail."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_scalar_example():
    """"Ring Attention: Distributed Reads with Online Softmax", section "Do not
    average independently normalized shard outputs": shard A (score 0, value
    0) and shard B (score 10, value 1)."""
    with open(os.path.join(GOLDEN, "scalar_two_shards.json")) as f:
        gold = json.load(f)
    a = (np.array([[gold["shard_a"]["value"]]]), np.array([gold["shard_a"]["score"]]))
    b = (np.array([[gold["shard_b"]["value"]]]), np.array([gold["shard_b"]["score"]]))
    o, lse = oracle.merge_lse(a, b)
    digits = gold["printed"]["global_softmax_output_digits"]
    assert round(float(o[0, 0]), digits) == gold["printed"]["global_softmax_output"]
    assert abs(float(lse[0]) - np.log(1 + np.exp(10.0))) <= 1e-12


def _stats(rng, rows, D):
    u = rng.standard_normal((rows, D))
    l = rng.uniform(0.5, 40.0, rows)
    m = rng.normal(0.0, 5.0, rows)
    return u, l, m


def test_equivalent_to_the_stats_merge():
    rng = np.random.default_rng(0)
    s1, s2 = _stats(rng, 50, 7), _stats(rng, 50, 7)
    # one row without keys on each side and one on both
    s1[1][3], s1[2][3] = 0.0, -np.inf
    s1[0][3] = 0.0
    s2[1][4], s2[2][4] = 0.0, -np.inf
    s2[0][4] = 0.0
    s1[1][5], s1[2][5], s1[0][5] = 0.0, -np.inf, 0.0
    s2[1][5], s2[2][5], s2[0][5] = 0.0, -np.inf, 0.0
    u, l, m = oracle.merge_stats(s1, s2)
    ref_o, ref_lse = oracle.normalize(u, l), oracle.stats_to_lse(m, l)
    def as_lse(st):
        return oracle.normalize(st[0], st[1]), oracle.stats_to_lse(st[2], st[1])
    o, lse = oracle.merge_lse(as_lse(s1), as_lse(s2))
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-12
    assert np.abs(o - ref_o).max() <= 1e-12
    assert np.all(o[~fin] == 0.0)


def test_closed_forms():
    o = np.array([[1.0, -2.0, 3.0]])
    # a block merged with itself: same output, lse + log 2
    mo, ml = oracle.merge_lse((o, np.array([1.5])), (o, np.array([1.5])))
    assert np.allclose(mo, o, atol=1e-15) and abs(ml[0] - (1.5 + np.log(2))) <= 1e-14
    # an empty side changes nothing
    mo, ml = oracle.merge_lse((o, np.array([0.25])), (np.zeros_like(o), np.array([-np.inf])))
    assert np.array_equal(mo, o) and ml[0] == 0.25


def test_merge_is_associative_and_commutative():
    rng = np.random.default_rng(1)
    blocks = [(rng.standard_normal((9, 4)), rng.normal(0, 3, 9)) for _ in range(3)]
    left = oracle.merge_lse(oracle.merge_lse(blocks[0], blocks[1]), blocks[2])
    right = oracle.merge_lse(blocks[0], oracle.merge_lse(blocks[2], blocks[1]))
    assert np.abs(left[0] - right[0]).max() <= 1e-12
    assert np.abs(left[1] - right[1]).max() <= 1e-12


def test_planted_mistake_fails():
    """Weighting by exp(lse) without renormalising is wrong."""
    rng = np.random.default_rng(2)
    a = (rng.standard_normal((5, 3)), rng.normal(0, 1, 5))
    b = (rng.standard_normal((5, 3)), rng.normal(0, 1, 5))
    good, _ = oracle.merge_lse(a, b)
    bad = np.exp(a[1])[:, None] * a[0] + np.exp(b[1])[:, None] * b[0]
    assert np.abs(bad - good).max() > 1e-2
