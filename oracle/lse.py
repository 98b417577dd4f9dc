"""Log-sum-exp form of the online-softmax merge, fp64 (test infrastructure,
same rule as ``oracle.attention``).

[GLOS] glossary entry "ring attention", "Online softmax": outputs of
different key/value blocks are combined with the log-sum-exp trick. With a
row's statistics (u, l, m) of the pages' merge, the normalised output is
O = u / l and its log-sum-exp lse = m + log(l): the log of the row's softmax
denominator in the units of the scaled scores. Two blocks combine as

    lse = log(exp(lse_a) + exp(lse_b))
    O   = exp(lse_a - lse) O_a + exp(lse_b - lse) O_b

A block with lse = -inf (it saw no key) weighs nothing; two such blocks give
O = 0, lse = -inf.
"""
from __future__ import annotations

import numpy as np


def stats_to_lse(m, l):
    """lse = m + log(l), -inf where l == 0."""
    m, l = np.asarray(m, dtype=np.float64), np.asarray(l, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)


def merge_lse(acc, new):
    """(O, lse) of the union of two blocks, from each block's (O, lse)."""
    oa, la = (np.asarray(x, dtype=np.float64) for x in acc)
    ob, lb = (np.asarray(x, dtype=np.float64) for x in new)
    mx = np.maximum(la, lb)
    empty = mx == -np.inf
    shift = np.where(empty, 0.0, mx)
    ea = np.where(la == -np.inf, 0.0, np.exp(la - shift))
    eb = np.where(lb == -np.inf, 0.0, np.exp(lb - shift))
    s = ea + eb
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(empty, -np.inf, shift + np.log(np.where(empty, 1.0, s)))
        wa = np.where(empty, 0.0, ea / np.where(empty, 1.0, s))
        wb = np.where(empty, 0.0, eb / np.where(empty, 1.0, s))
    return wa[..., None] * oa + wb[..., None] * ob, lse
