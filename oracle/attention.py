"""Plain fp64 CPU oracle for the chunked (ring) forward pass of softmax attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) may import or
run anything in this package. The library's product path (the CUDA kernels,
the C ABI and the Python binding) never imports it, and it never imports the
library: the two share no code. Inputs come in as plain arrays; every value is
upcast exactly to float64 before any arithmetic.

Sources (web pages; cited by title and section):

* [EX]  Ring-attention exercise page "systems-distributed-ring-attention-online-
        softmax": task statement (the three functions, their outputs, and the
        requirement that the result not depend on how the keys are split,
        down to chunks of one key) and its two hints (max subtraction; the
        exp(own_max - new_max) rescale).
* [BLOG] "Ring Attention: Distributed Reads with Online Softmax":
        sections "Partition the sequence across devices", "Do not average
        independently normalized shard outputs", "A simple forward schedule",
        "Causal masks depend on global positions", "Try it".
* [GLOS] Glossary entry "ring attention": algorithm steps (1)-(6) and the
        "Online softmax" paragraph.

Conventions (readings of what the pages leave open; each is listed in the
design notes):

* q: [B, Hq, Sq, D]; k, v: [B, Hkv, Sk, D]; Hq % Hkv == 0 and query head h
  reads key/value head h // (Hq // Hkv) (grouped heads; the pages do not
  discuss head sharing, this is the plainest grouping).
* Scores are s_ij = scale * <q_i, k_j>; the returned row max m is in those
  scaled, natural-log units, and l = sum_j exp(s_ij - m).
* Causal: key j is visible to query i iff pos_k[j] <= pos_q[i], with GLOBAL
  positions ([BLOG] "Causal masks depend on global positions").
* A row that sees no key has u = 0, l = 0, m = -inf, and its output is 0.
  In a merge a side with m = -inf contributes nothing (no exp(-inf + inf)).
* Documents (packed variable-length sequences; the pages do not treat them,
  this is the plainest extension of the global-position mask): ``docs`` is a
  strictly increasing list of boundaries b_0 < b_1 < ... < b_n, document d
  holds the positions [b_d, b_{d+1}), and a key is visible to a query only if
  both lie in the same document (and, when causal, the key is not in the
  query's future). ``docs=None`` is one document holding every position.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def document_of(pos, docs):
    """Index d of the document [b_d, b_{d+1}) that holds each position.

    Raises ValueError for a position outside [b_0, b_n) or for boundaries
    that are not strictly increasing.
    """
    pos = np.asarray(pos, dtype=np.int64)
    b = np.asarray(docs, dtype=np.int64)
    if b.ndim != 1 or b.size < 2 or (np.diff(b) <= 0).any():
        raise ValueError("document boundaries must be >= 2 strictly increasing values")
    d = np.searchsorted(b, pos, side="right") - 1
    if pos.size and ((d < 0).any() or (d >= b.size - 1).any()):
        raise ValueError("a position lies outside every document")
    return d


def _visible(q_pos, k_pos, causal, docs=None):
    """Boolean [Sq, Sk] visibility matrix from global positions.

    [BLOG] "Causal masks depend on global positions": a query may not read a
    key that lies in its future, judged by global position, not by local
    row/column index. With documents, also only keys of the query's own
    document (the module's reading).
    """
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    if not causal:
        vis = np.ones((q_pos.shape[0], k_pos.shape[0]), dtype=bool)
    else:
        vis = k_pos[None, :] <= q_pos[:, None]
    if docs is not None:
        vis &= document_of(q_pos, docs)[:, None] == document_of(k_pos, docs)[None, :]
    return vis


def _head_group(Hq, Hkv):
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError(f"Hq={Hq} must be a positive multiple of Hkv={Hkv}")
    return Hq // Hkv


def chunk_stats(q, k, v, q_pos, k_pos, causal, scale, docs=None):
    """Statistics of one key/value chunk, computed as if it were the only one.

    [EX] task statement: returns (chunk_output, chunk_sum, chunk_max) = the
    un-normalised weighted value sum u, the un-normalised softmax denominator
    l, and the row-wise max score m. [EX] first hint: the same max-subtraction
    as scaled dot-product attention, with numerator and denominator returned
    separately instead of divided.

    Returns u [B, Hq, Sq, D], l [B, Hq, Sq], m [B, Hq, Sq] (float64).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    g = _head_group(Hq, Hkv)
    vis = _visible(q_pos, k_pos, causal, docs)
    u = np.zeros((B, Hq, Sq, v.shape[3]))
    l = np.zeros((B, Hq, Sq))
    m = np.full((B, Hq, Sq), NEG_INF)
    if Sk == 0 or Sq == 0:
        return u, l, m
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, h // g], v[b, h // g]
            s = scale * (q[b, h] @ kh.T)                  # [Sq, Sk] scores
            s = np.where(vis, s, NEG_INF)
            mrow = s.max(axis=1)                          # -inf if nothing visible
            shift = np.where(np.isfinite(mrow), mrow, 0.0)
            w = np.exp(s - shift[:, None])                # exp(-inf) = 0
            u[b, h] = w @ vh
            l[b, h] = w.sum(axis=1)
            m[b, h] = mrow
    return u, l, m


def merge_stats(acc, new):
    """Online-softmax merge of two sets of statistics.

    [EX] task statement and second hint: the shared max is
    max(acc_max, chunk_max); BOTH sides are multiplied by
    exp(own_max - new_max) before their numerators and denominators are added;
    stats relative to different maxes are never added directly.
    [BLOG] "Do not average ...": keep m, l and u per shard and merge them.

    A side whose max is -inf (it saw no key) contributes zero.
    """
    u1, l1, m1 = (_f64(x) for x in acc)
    u2, l2, m2 = (_f64(x) for x in new)
    m = np.maximum(m1, m2)
    with np.errstate(invalid="ignore"):
        a1 = np.where(m1 == NEG_INF, 0.0, np.exp(m1 - m))
        a2 = np.where(m2 == NEG_INF, 0.0, np.exp(m2 - m))
    u = a1[..., None] * u1 + a2[..., None] * u2
    l = a1 * l1 + a2 * l2
    return u, l, m


def normalize(u, l):
    """Final output u / l ([BLOG] "A simple forward schedule", last step).

    A row with l == 0 saw no key; its output is 0 (a reading: the pages do
    not define it).
    """
    u, l = _f64(u), _f64(l)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l[..., None] > 0, u / np.where(l > 0, l, 1.0)[..., None], 0.0)
    return o


def full_attention(q, k, v, q_pos, k_pos, causal, scale, docs=None):
    """Ordinary softmax attention over the whole key/value sequence at once.

    This is the plain definition the chunked method must equal exactly: the
    [EX] task statement asks for the result of ordinary attention over all
    key/value chunks joined into one sequence. Per row: m = max of visible
    scaled scores, l = sum exp(s - m), O = sum exp(s - m) v / l.

    Returns O [B, Hq, Sq, D], m [B, Hq, Sq], l [B, Hq, Sq].
    """
    u, l, m = chunk_stats(q, k, v, q_pos, k_pos, causal, scale, docs)
    return normalize(u, l), m, l


def ring_order(rank, world):
    """Chunk visited by device ``rank`` at each ring step.

    [BLOG] "Partition the sequence across devices": each device sends its
    shard to the next device and receives one from its predecessor, so at step
    s device r holds the shard that started on device (r - s) mod P.
    [GLOS] algorithm steps (1)-(5): step 0 is the device's own chunk.
    """
    return [(rank - s) % world for s in range(world)]


def ring_attention(q, k_chunks, v_chunks, q_pos, k_pos_chunks, causal, scale,
                   order=None, docs=None):
    """The pages' chunked algorithm, written out: stats per chunk + merges.

    [EX] task statement: visit key/value chunks one at a time, never forming
    the full attention matrix. [BLOG] "A simple forward schedule": initialise
    a running summary, for each shard compute its contribution and merge it,
    finally normalise u / l. ``order`` lists the chunk indices to visit
    (default: index order). Returns O, m, l like ``full_attention``.

    This second path exists to check the pages' claims against the definition
    (chunk invariance, merge correctness); parity tests of the CUDA path
    compare against ``full_attention`` / ``attention_rows``.
    """
    q = _f64(q)
    B, Hq, Sq, _ = q.shape
    D = _f64(v_chunks[0]).shape[3] if len(v_chunks) else q.shape[3]
    acc = (np.zeros((B, Hq, Sq, D)), np.zeros((B, Hq, Sq)),
           np.full((B, Hq, Sq), NEG_INF))
    if order is None:
        order = range(len(k_chunks))
    for c in order:
        st = chunk_stats(q, k_chunks[c], v_chunks[c], q_pos, k_pos_chunks[c],
                         causal, scale, docs)
        acc = merge_stats(acc, st)
    u, l, m = acc
    return normalize(u, l), m, l


def attention_rows(q, k, v, q_pos, k_pos, causal, scale, rows, docs=None):
    """The definition of ``full_attention`` evaluated for selected rows only.

    ``rows`` is a list of (b, h, i) triples. Each row is computed on its own,
    exactly against all of its visible keys, so that sampled rows of very long
    sequences can be checked without forming [Sq, Sk] matrices. Inputs may be
    any array type convertible to float64 (per head slices are upcast lazily).

    Returns arrays O [R, D], m [R], l [R] in the order of ``rows``.
    """
    rows = list(rows)
    Hq = q.shape[1]
    Hkv = k.shape[1]
    g = _head_group(Hq, Hkv)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    D = v.shape[3]
    O = np.zeros((len(rows), D))
    M = np.full(len(rows), NEG_INF)
    L = np.zeros(len(rows))
    if k.shape[2] == 0:
        return O, M, L
    by_head = {}
    for idx, (b, h, i) in enumerate(rows):
        by_head.setdefault((b, h // g), []).append((idx, h, i))
    for (b, hk), items in by_head.items():
        kh = _f64(k[b, hk])
        vh = _f64(v[b, hk])
        # rows are independent: evaluate a group of them with one product
        for g0 in range(0, len(items), 32):
            grp = items[g0:g0 + 32]
            idx = np.array([it[0] for it in grp])
            qs = np.stack([_f64(q[b, h, i]) for _, h, i in grp])     # [R, D]
            s = scale * (qs @ kh.T)                                  # [R, Sk]
            qp = np.array([q_pos[i] for _, _, i in grp])
            s = np.where(_visible(qp, k_pos, causal, docs), s, NEG_INF)
            mrow = s.max(axis=1)
            seen = np.isfinite(mrow)
            shift = np.where(seen, mrow, 0.0)
            w = np.exp(s - shift[:, None])
            lrow = w.sum(axis=1)
            num = w @ vh
            O[idx] = np.where(seen[:, None], num / np.where(seen, lrow, 1.0)[:, None], 0.0)
            M[idx] = mrow
            L[idx] = np.where(seen, lrow, 0.0)
    return O, M, L


def unmasked_pairs(q_pos, k_pos, causal, docs=None):
    """Exact number of visible (query, key) pairs: the work a causal mask
    leaves ([BLOG] "Separate local compute from network traffic": attention
    arithmetic counts query-key pairs). With documents, a query counts the
    keys of its own document only (up to its position when causal)."""
    q_pos = np.sort(np.asarray(q_pos, dtype=np.int64))
    k_pos = np.sort(np.asarray(k_pos, dtype=np.int64))
    if docs is None:
        if not causal:
            return int(q_pos.size) * int(k_pos.size)
        return int(np.searchsorted(k_pos, q_pos, side="right").sum())
    b = np.asarray(docs, dtype=np.int64)
    d = document_of(q_pos, b)
    document_of(k_pos, b)
    lo = np.searchsorted(k_pos, b[d], side="left")
    if causal:
        hi = np.searchsorted(k_pos, q_pos, side="right")
    else:
        hi = np.searchsorted(k_pos, b[d + 1], side="left")
    return int((hi - lo).sum())
