"""Sequence layouts over P devices (or P virtual ranks on one GPU).

Each layout assigns every global position to exactly one rank and is described
by position spans (len, pos0, step), the form the C ABI takes:

* contiguous: rank r holds n/P consecutive positions ("Ring Attention:
  Distributed Reads with Online Softmax", "Partition the sequence across
  devices").
* zigzag: the sequence is cut into 2P blocks; rank r holds block r and block
  2P-1-r, pairing an early block with a late one (same blog, "Causal masks
  depend on global positions": paired early/late chunks balance causal work).
* striped: rank r holds positions r, r+P, r+2P, ... (glossary "ring
  attention", "Variants (1) striped attention").
"""
from __future__ import annotations

import torch


def rank_spans(kind: str, n: int, P: int):
    """List over ranks of span lists [(len, pos0, step), ...]."""
    if kind == "contiguous":
        if n % P:
            raise ValueError("n must be a multiple of P")
        w = n // P
        return [[(w, r * w, 1)] for r in range(P)]
    if kind == "zigzag":
        if n % (2 * P):
            raise ValueError("n must be a multiple of 2P")
        w = n // (2 * P)
        return [[(w, r * w, 1), (w, (2 * P - 1 - r) * w, 1)] for r in range(P)]
    if kind == "striped":
        if n % P:
            raise ValueError("n must be a multiple of P")
        return [[(n // P, r, P)] for r in range(P)]
    raise ValueError(f"unknown layout {kind!r}")


def span_positions(spans) -> torch.Tensor:
    """Global positions of consecutive rows described by spans."""
    parts = [torch.arange(p0, p0 + st * ln, st, dtype=torch.int64) if ln else
             torch.empty(0, dtype=torch.int64) for ln, p0, st in spans]
    return torch.cat(parts) if parts else torch.empty(0, dtype=torch.int64)


def permutation(kind: str, n: int, P: int) -> torch.Tensor:
    """Global position of each row in rank-major storage order."""
    return torch.cat([span_positions(s) for s in rank_spans(kind, n, P)])


def shard(x: torch.Tensor, kind: str, P: int, dim: int = 2):
    """Split a global-order tensor into P per-rank contiguous shards."""
    n = x.shape[dim]
    out = []
    for spans in rank_spans(kind, n, P):
        idx = span_positions(spans).to(x.device)
        out.append(x.index_select(dim, idx).contiguous())
    return out


def to_global(x_rank_major: torch.Tensor, kind: str, P: int, dim: int = 2) -> torch.Tensor:
    """Inverse of concatenating ``shard`` outputs: back to global order."""
    perm = permutation(kind, x_rank_major.shape[dim], P).to(x_rank_major.device)
    out = torch.empty_like(x_rank_major)
    out.index_copy_(dim, perm, x_rank_major)
    return out
