"""Plain fp64 CPU oracle for the backward pass of softmax attention.

TEST INFRASTRUCTURE (same rule as ``oracle.attention``): imported only by
tests/, ``__graft_entry__.smoke()`` and bench.py's CPU legs. It shares no code
with the library.

Source: [BLOG] "Ring Attention: Distributed Reads with Online Softmax",
section "Backward must aggregate shared dependencies": a query's gradient
reaches the keys and values of every shard it attended to; those
contributions are summed per key/value shard and returned to its owner;
recomputed probability tiles must use the forward's scaling and masks; the
distributed gradients are to be checked against a single-device reference.

The definition is the chain rule through O = softmax(S) V with
S = scale * Q K^T over the visible keys (global positions, as in the forward):

    P  = softmax(S)                 (a row that sees no key: P = 0, O = 0)
    dV = P^T dO
    dP = dO V^T
    dS = P * (dP - rowsum(P * dP))  (Jacobian of the row softmax)
    dQ = scale * dS K
    dK = scale * dS^T Q

With grouped heads, key/value head g receives the sum over the query heads
h with h // (Hq / Hkv) == g (the forward's head mapping). ``docs`` restricts
visibility to the query's own document, as in the forward.
"""
from __future__ import annotations

import numpy as np

from .attention import _f64, _head_group, _visible, full_attention


def attention_backward(q, k, v, dout, q_pos, k_pos, causal, scale, docs=None):
    """Gradients of sum(dout * O) with respect to q, k, v, by the definition.

    Shapes: q, dout [B, Hq, Sq, D]; k, v [B, Hkv, Sk, D]. Returns dq, dk, dv
    (float64) of the shapes of q, k, v.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    g = _head_group(Hq, Hkv)
    vis = _visible(q_pos, k_pos, causal, docs)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    if Sq == 0 or Sk == 0:
        return dq, dk, dv
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, h // g], v[b, h // g]
            s = np.where(vis, scale * (q[b, h] @ kh.T), -np.inf)
            mrow = s.max(axis=1)
            seen = np.isfinite(mrow)
            w = np.exp(s - np.where(seen, mrow, 0.0)[:, None])
            lrow = w.sum(axis=1)
            p = np.where(seen[:, None], w / np.where(seen, lrow, 1.0)[:, None], 0.0)
            dp = dout[b, h] @ vh.T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dv[b, h // g] += p.T @ dout[b, h]
            dq[b, h] = scale * (ds @ kh)
            dk[b, h // g] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


def ring_attention_backward(q, k_chunks, v_chunks, dout, q_pos, k_pos_chunks, causal, scale,
                            docs=None):
    """The blog's aggregation, chunk by chunk.

    The forward's row statistics (max m and denominator l over ALL chunks)
    fix P; for each key/value chunk its probability tile is recomputed with
    them, P_c = exp(S_c - m) / l, under the same scale and mask. The chunk's
    own gradients dK_c, dV_c are complete after that one visit (every query
    row's contribution is summed into them, for the chunk's owner); dQ
    accumulates over the chunks. The row term rowsum(P * dP) is taken in its
    equivalent form rowsum(dO * O) (sum over all chunks of P_c * dP_c equals
    dO . O, since O = sum_c P_c V_c), which is what a shard can compute without
    seeing the other shards.

    Returns dq [B, Hq, Sq, D] and the lists dk_chunks, dv_chunks.
    """
    q, dout = _f64(q), _f64(dout)
    B, Hq, Sq, D = q.shape
    k_all = np.concatenate([_f64(x) for x in k_chunks], axis=2)
    v_all = np.concatenate([_f64(x) for x in v_chunks], axis=2)
    k_pos_all = np.concatenate([np.asarray(p, dtype=np.int64) for p in k_pos_chunks])
    O, m, l = full_attention(q, k_all, v_all, q_pos, k_pos_all, causal, scale, docs)
    delta = (dout * O).sum(axis=3)                       # [B, Hq, Sq]
    Hkv = k_all.shape[1]
    g = _head_group(Hq, Hkv)
    seen = np.isfinite(m)
    shift = np.where(seen, m, 0.0)
    lsafe = np.where(seen, l, 1.0)
    dq = np.zeros_like(q)
    dk_chunks, dv_chunks = [], []
    for kc, vc, kp in zip(k_chunks, v_chunks, k_pos_chunks):
        kc, vc = _f64(kc), _f64(vc)
        vis = _visible(q_pos, kp, causal, docs)
        dkc = np.zeros_like(kc)
        dvc = np.zeros_like(vc)
        for b in range(B):
            for h in range(Hq):
                s = np.where(vis, scale * (q[b, h] @ kc[b, h // g].T), -np.inf)
                p = np.exp(s - shift[b, h][:, None]) / lsafe[b, h][:, None]
                p = np.where(seen[b, h][:, None], p, 0.0)
                dp = dout[b, h] @ vc[b, h // g].T
                ds = p * (dp - delta[b, h][:, None])
                dvc[b, h // g] += p.T @ dout[b, h]
                dkc[b, h // g] += scale * (ds.T @ q[b, h])
                dq[b, h] += scale * (ds @ kc[b, h // g])
        dk_chunks.append(dkc)
        dv_chunks.append(dvc)
    return dq, dk_chunks, dv_chunks


def gradient_rounding_bounds(q, k, v, dout, q_pos, k_pos, causal, scale, docs=None,
                             u=2.0 ** -8):
    """Elementwise bounds on the rounding error of a backward that rounds the
    probabilities P and the score gradients dS to a number format of unit
    roundoff ``u`` (bf16: 2^-8) before multiplying them, given the exact row
    statistics and O, and accumulates the products in fp32.

    This is the tolerance of the parity tests, derived from that arithmetic;
    it is not part of the method. With the exact P, dS of the definition and
    their rounded forms P~, dS~ (|P~ - P| <= u P, |dS~ - dS| <= u |dS|):

        |dV~ - dV| <= u P^T |dO|
        |dQ~ - dQ| <= scale u |dS| |K|
        |dK~ - dK| <= scale u |dS|^T |Q|

    (the fp32 parts -- the scores, exp2, the row term, the accumulation --
    contribute errors some thousand times smaller). With grouped heads the
    key/value bounds add up over the group's query heads, like the gradients.
    Returns (bdq, bdk, bdv) of the shapes of q, k, v.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    g = _head_group(Hq, Hkv)
    vis = _visible(q_pos, k_pos, causal, docs)
    bdq, bdk, bdv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    if Sq == 0 or k.shape[2] == 0:
        return bdq, bdk, bdv
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, h // g], v[b, h // g]
            s = np.where(vis, scale * (q[b, h] @ kh.T), -np.inf)
            mrow = s.max(axis=1)
            seen = np.isfinite(mrow)
            w = np.exp(s - np.where(seen, mrow, 0.0)[:, None])
            lrow = w.sum(axis=1)
            p = np.where(seen[:, None], w / np.where(seen, lrow, 1.0)[:, None], 0.0)
            dp = dout[b, h] @ vh.T
            ads = np.abs(p * (dp - (p * dp).sum(axis=1, keepdims=True)))
            bdv[b, h // g] += u * (p.T @ np.abs(dout[b, h]))
            bdq[b, h] = scale * u * (ads @ np.abs(kh))
            bdk[b, h // g] += scale * u * (ads.T @ np.abs(q[b, h]))
    return bdq, bdk, bdv
