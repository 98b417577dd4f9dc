"""Global positions owned by each device under the pages' sequence layouts.

TEST INFRASTRUCTURE (same rule as ``oracle.attention``): imported only by
tests, smoke() and bench.py's CPU legs.

* contiguous: [BLOG] "Partition the sequence across devices": device r holds
  roughly n/P consecutive positions.
* zigzag: [BLOG] "Causal masks depend on global positions": pairing an early
  chunk with a late one balances causal work. Reading: the sequence is cut into
  2P equal blocks and device r owns block r followed by block 2P-1-r.
* striped: [GLOS] "Variants (1) Striped attention": tokens are reordered so
  each chunk holds positions from all over the sequence. Reading: device r
  owns positions r, r+P, r+2P, ...

Each function returns a list of P int64 arrays, device r's positions in the
order its rows are stored.
"""
from __future__ import annotations

import numpy as np


def contiguous(n, P):
    if n % P:
        raise ValueError("n must be a multiple of P")
    w = n // P
    return [np.arange(r * w, (r + 1) * w, dtype=np.int64) for r in range(P)]


def zigzag(n, P):
    if n % (2 * P):
        raise ValueError("n must be a multiple of 2P")
    w = n // (2 * P)
    out = []
    for r in range(P):
        early = np.arange(r * w, (r + 1) * w, dtype=np.int64)
        late_block = 2 * P - 1 - r
        late = np.arange(late_block * w, (late_block + 1) * w, dtype=np.int64)
        out.append(np.concatenate([early, late]))
    return out


def striped(n, P):
    if n % P:
        raise ValueError("n must be a multiple of P")
    return [np.arange(r, n, P, dtype=np.int64) for r in range(P)]


LAYOUTS = {"contiguous": contiguous, "zigzag": zigzag, "striped": striped}


def positions(kind, n, P):
    return LAYOUTS[kind](n, P)
