"""Torch-facing binding of the C ABI: same operations, tensors in and out.

Only argument marshalling happens here (pointers, strides, spans, the current
CUDA stream). Every step of the computation runs in the library's kernels;
PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib
from ._lib import KvChunk, Problem, QSegment, Strides, check, load, positions

Span = tuple  # (len, pos0, step)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.RA_BF16
    if t.dtype == torch.float32:
        return _lib.RA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use bfloat16 or float32")


def _strides(t: torch.Tensor) -> Strides:
    if t.dim() != 4:
        raise ValueError("tensors are [batch, head, row, head_dim]")
    if t.shape[3] > 1 and t.stride(3) != 1:
        raise ValueError("head_dim must be contiguous")
    return Strides(t.stride(0), t.stride(1), t.stride(2))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_cuda(t: torch.Tensor, what: str):
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")


def _segments(q: torch.Tensor, q_segments):
    Sq = q.shape[2]
    if q_segments is None:
        q_segments = [(Sq, [(Sq, 0, 1)])]
    arr = (QSegment * max(1, len(q_segments)))()
    for i, (ln, spans) in enumerate(q_segments):
        arr[i].len = int(ln)
        arr[i].pos = positions(spans)
    return arr, len(q_segments)


def _chunks(k_chunks, v_chunks, chunk_spans, host=False):
    if len(k_chunks) != len(v_chunks):
        raise ValueError("need as many value chunks as key chunks")
    if chunk_spans is None:
        chunk_spans, p = [], 0
        for k in k_chunks:
            chunk_spans.append([(k.shape[2], p, 1)])
            p += k.shape[2]
    arr = (KvChunk * max(1, len(k_chunks)))()
    for i, (k, v) in enumerate(zip(k_chunks, v_chunks)):
        if not host:
            _check_cuda(k, "k"); _check_cuda(v, "v")
        if k.shape != v.shape:
            raise ValueError("k and v chunks must have the same shape")
        arr[i].k = k.data_ptr()
        arr[i].v = v.data_ptr()
        arr[i].len = k.shape[2]
        arr[i].k_strides = _strides(k)
        arr[i].v_strides = _strides(v)
        arr[i].pos = positions(chunk_spans[i])
    return arr, len(k_chunks)


def _set_docs(pb, docs):
    """Document boundaries b_0 < ... < b_n (host int64 array kept alive on pb)."""
    if docs is None:
        pb.n_docs = 0
        pb.doc_bounds = None
        return
    b = [int(x) for x in docs]
    if len(b) < 2:
        raise ValueError("docs needs at least two boundaries (one document)")
    arr = (ctypes.c_int64 * len(b))(*b)
    pb._docs_keepalive = arr
    pb.doc_bounds = ctypes.cast(arr, ctypes.c_void_p)
    pb.n_docs = len(b) - 1


def _problem(q, Hkv, causal, scale, out_strides, docs=None):
    B, Hq, Sq, D = q.shape
    pb = Problem()
    pb.B, pb.Hq, pb.Hkv, pb.D, pb.Sq = B, Hq, Hkv, D, Sq
    pb.dtype = _dtype_code(q)
    pb.causal = 1 if causal else 0
    pb.scale = float(scale) if scale is not None else 0.0
    pb.o_fp32 = 0
    pb.q_strides = _strides(q)
    pb.o_strides = out_strides
    _set_docs(pb, docs)
    return pb


def ring_attention(q, k_chunks, v_chunks, *, chunk_spans=None, q_segments=None,
                   causal=False, scale=None, out=None, m=None, l=None, out_dtype=None,
                   docs=None, stream=None):
    """Chunked forward pass over key/value chunks (one persistent kernel).

    q: [B, Hq, Sq, D] (bf16 or fp32, CUDA). k_chunks / v_chunks: lists of
    [B, Hkv, len_c, D]. chunk_spans[c]: global positions of chunk c as spans
    (default: the chunks concatenated in list order from position 0).
    q_segments: list of (len, spans) splitting Q's rows (default: one segment
    at positions 0..Sq-1); with as many segments as chunks, segment r walks
    the chunks in ring order starting at chunk r.
    out_dtype: torch.float32 to receive O in fp32 from bf16 inputs (default:
    the dtype of q, or of ``out`` when given).
    docs: packed documents, boundaries b_0 < ... < b_n of global positions
    (a query sees only keys of its own document [b_d, b_{d+1})).
    Returns (O [B, Hq, Sq, D], m [B, Hq, Sq] fp32, l [B, Hq, Sq] fp32).
    """
    lib = load()
    _check_cuda(q, "q")
    B, Hq, Sq, D = q.shape
    Hkv = k_chunks[0].shape[1] if k_chunks else Hq
    if out is None:
        out = torch.empty(q.shape, device=q.device, dtype=out_dtype or q.dtype)
    if out.dtype not in (q.dtype, torch.float32):
        raise TypeError("O must have the dtype of q or float32")
    if m is None:
        m = torch.empty(B, Hq, Sq, device=q.device, dtype=torch.float32)
    if l is None:
        l = torch.empty(B, Hq, Sq, device=q.device, dtype=torch.float32)
    pb = _problem(q, Hkv, causal, scale, _strides(out), docs)
    pb.o_fp32 = 1 if (out.dtype == torch.float32 and q.dtype != torch.float32) else 0
    segs, nsegs = _segments(q, q_segments)
    chs, nch = _chunks(k_chunks, v_chunks, chunk_spans)
    check(lib.ra_ring_attention(ctypes.byref(pb), q.data_ptr(), segs, nsegs, chs, nch,
                                out.data_ptr(), m.data_ptr(), l.data_ptr(), _stream(stream)))
    return out, m, l


def ring_attention_host(q, k_chunks, v_chunks, *, chunk_spans=None, q_segments=None,
                        causal=False, scale=None, out=None, m=None, l=None, out_dtype=None,
                        docs=None, stream=None):
    """ring_attention with every tensor in host memory (pinned for full speed).

    The library copies the inputs to the device, runs the ring kernel and
    copies O, m, l back, all enqueued on ``stream`` (default: the current CUDA
    stream). The results are valid, and the inputs may be changed, only after
    that stream has been synchronised. All tensors must be contiguous CPU
    tensors; calls on different streams overlap copies with kernels.
    Returns (O, m, l) as host tensors.
    """
    lib = load()
    for t in [q, *k_chunks, *v_chunks]:
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("ring_attention_host takes contiguous CPU tensors")
    B, Hq, Sq, D = q.shape
    Hkv = k_chunks[0].shape[1] if k_chunks else Hq
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, pin_memory=pin)
    if out.dtype not in (q.dtype, torch.float32):
        raise TypeError("O must have the dtype of q or float32")
    if m is None:
        m = torch.empty(B, Hq, Sq, dtype=torch.float32, pin_memory=pin)
    if l is None:
        l = torch.empty(B, Hq, Sq, dtype=torch.float32, pin_memory=pin)
    for t in (out, m, l):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("outputs must be contiguous CPU tensors")
    pb = _problem(q, Hkv, causal, scale, _strides(out), docs)
    pb.o_fp32 = 1 if (out.dtype == torch.float32 and q.dtype != torch.float32) else 0
    segs, nsegs = _segments(q, q_segments)
    chs, nch = _chunks(k_chunks, v_chunks, chunk_spans, host=True)
    check(lib.ra_ring_attention_host(ctypes.byref(pb), q.data_ptr(), segs, nsegs, chs, nch,
                                     out.data_ptr(), m.data_ptr(), l.data_ptr(), _stream(stream)))
    return out, m, l


def ring_attention_bwd(q, k_chunks, v_chunks, o, dout, m, l, *, chunk_spans=None,
                       q_segments=None, causal=False, scale=None, dq=None, dk=None, dv=None,
                       docs=None, stream=None):
    """Gradients of ``ring_attention``'s O: (dq, [dk per chunk], [dv per chunk]).

    q, k_chunks, v_chunks, chunk_spans, q_segments, causal, scale, docs:
    exactly as given to the forward call; o, m, l: its outputs; dout: bf16 gradient of O
    with o's strides. Gradients are fp32: dq like q, dk/dv like each chunk
    (dense). bf16 inputs only.
    """
    lib = load()
    for t in (q, o, dout, m, l):
        _check_cuda(t, "tensors")
    if dout.shape != o.shape or dout.stride() != o.stride():
        raise ValueError("dout must have o's shape and strides")
    if dout.dtype != torch.bfloat16:
        raise TypeError("dout must be bfloat16")
    B, Hq, Sq, D = q.shape
    Hkv = k_chunks[0].shape[1] if k_chunks else Hq
    if dq is None:
        dq = torch.empty(B, Hq, Sq, D, device=q.device, dtype=torch.float32)
    if dk is None:
        dk = [torch.empty(k.shape, device=q.device, dtype=torch.float32) for k in k_chunks]
    if dv is None:
        dv = [torch.empty(v.shape, device=q.device, dtype=torch.float32) for v in v_chunks]
    for t in [dq, *dk, *dv]:
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("gradients are dense fp32 tensors")
    pb = _problem(q, Hkv, causal, scale, _strides(o), docs)
    pb.o_fp32 = 1 if (o.dtype == torch.float32 and q.dtype != torch.float32) else 0
    segs, nsegs = _segments(q, q_segments)
    chs, nch = _chunks(k_chunks, v_chunks, chunk_spans)
    grads = (_lib.KvGrad * max(1, nch))()
    for i in range(nch):
        grads[i].dk = dk[i].data_ptr()
        grads[i].dv = dv[i].data_ptr()
    check(lib.ra_ring_attention_bwd(ctypes.byref(pb), q.data_ptr(), segs, nsegs, chs, nch,
                                    o.data_ptr(), dout.data_ptr(), m.data_ptr(), l.data_ptr(),
                                    dq.data_ptr(), grads, _stream(stream)))
    return dq, dk, dv


def chunk_stats(q, k, v, *, spans=None, q_segments=None, causal=False, scale=None,
                u=None, l=None, m=None, docs=None, stream=None):
    """(u, l, m) of one key/value chunk, as if it were the only one.

    u: [B, Hq, Sq, D] fp32 un-normalised numerator; l, m: [B, Hq, Sq] fp32.
    spans: global positions of the chunk's rows (default 0..len-1).
    """
    lib = load()
    _check_cuda(q, "q")
    B, Hq, Sq, D = q.shape
    if u is None:
        u = torch.empty(B, Hq, Sq, D, device=q.device, dtype=torch.float32)
    if l is None:
        l = torch.empty(B, Hq, Sq, device=q.device, dtype=torch.float32)
    if m is None:
        m = torch.empty(B, Hq, Sq, device=q.device, dtype=torch.float32)
    pb = _problem(q, k.shape[1], causal, scale, _strides(u), docs)
    segs, nsegs = _segments(q, q_segments)
    chs, _ = _chunks([k], [v], None if spans is None else [spans])
    check(lib.ra_chunk_stats(ctypes.byref(pb), q.data_ptr(), segs, nsegs, chs,
                             u.data_ptr(), l.data_ptr(), m.data_ptr(), _stream(stream)))
    return u, l, m


def merge_stats(u_acc, l_acc, m_acc, u_new, l_new, m_new, stream=None):
    """In-place online-softmax merge of (u_new, l_new, m_new) into the accumulator."""
    lib = load()
    for t in (u_acc, l_acc, m_acc, u_new, l_new, m_new):
        _check_cuda(t, "stats")
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("statistics must be contiguous fp32 tensors")
    D = u_acc.shape[-1]
    rows = u_acc.numel() // D
    if u_new.numel() != u_acc.numel() or l_acc.numel() != rows or m_acc.numel() != rows \
            or l_new.numel() != rows or m_new.numel() != rows:
        raise ValueError("shape mismatch between the two sets of statistics")
    check(lib.ra_merge_stats(rows, D, u_acc.data_ptr(), l_acc.data_ptr(), m_acc.data_ptr(),
                             u_new.data_ptr(), l_new.data_ptr(), m_new.data_ptr(),
                             _stream(stream)))
    return u_acc, l_acc, m_acc


def merge_lse(o_acc, lse_acc, o_new, lse_new, stream=None):
    """In-place log-sum-exp merge of (o_new, lse_new) into (o_acc, lse_acc)."""
    lib = load()
    for t in (o_acc, lse_acc, o_new, lse_new):
        _check_cuda(t, "lse merge")
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("outputs and log-sum-exps must be contiguous fp32 tensors")
    D = o_acc.shape[-1]
    rows = o_acc.numel() // D
    if o_new.numel() != o_acc.numel() or lse_acc.numel() != rows or lse_new.numel() != rows:
        raise ValueError("shape mismatch between the two outputs")
    check(lib.ra_merge_lse(rows, D, o_acc.data_ptr(), lse_acc.data_ptr(), o_new.data_ptr(),
                           lse_new.data_ptr(), _stream(stream)))
    return o_acc, lse_acc


def stats_to_lse(m, l, lse=None, stream=None):
    """lse = m + log(l) per row (-inf where l = 0)."""
    lib = load()
    for t in (m, l):
        _check_cuda(t, "statistics")
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("statistics must be contiguous fp32 tensors")
    if lse is None:
        lse = torch.empty_like(m)
    check(lib.ra_stats_to_lse(m.numel(), m.data_ptr(), l.data_ptr(), lse.data_ptr(), _stream(stream)))
    return lse


def segment_work(B, Hq, Hkv, D, q_segments, chunk_lens, chunk_spans, causal, dtype=_lib.RA_BF16,
                 docs=None):
    """Per query segment: visible (query, key) pairs per head and scheduled
    128x128 tile products (host-side bookkeeping, no GPU needed)."""
    lib = load()
    Sq = sum(int(n) for n, _ in q_segments)
    pb = Problem()
    pb.B, pb.Hq, pb.Hkv, pb.D, pb.Sq = B, Hq, Hkv, D, Sq
    pb.dtype, pb.causal, pb.scale, pb.o_fp32 = dtype, 1 if causal else 0, 0.0, 0
    pb.q_strides = Strides(Hq * Sq * D, Sq * D, D)
    pb.o_strides = pb.q_strides
    _set_docs(pb, docs)
    segs = (QSegment * len(q_segments))()
    for i, (ln, spans) in enumerate(q_segments):
        segs[i].len = int(ln)
        segs[i].pos = positions(spans)
    chs = (KvChunk * max(1, len(chunk_lens)))()
    for i, (ln, spans) in enumerate(zip(chunk_lens, chunk_spans)):
        chs[i].len = int(ln)
        chs[i].pos = positions(spans)
    pairs = (ctypes.c_int64 * len(q_segments))()
    tiles = (ctypes.c_int64 * len(q_segments))()
    check(lib.ra_segment_work(ctypes.byref(pb), segs, len(q_segments), chs, len(chunk_lens),
                              ctypes.cast(pairs, ctypes.c_void_p),
                              ctypes.cast(tiles, ctypes.c_void_p)))
    return list(pairs), list(tiles)


def device_status(stream=None):
    """Synchronise ``stream`` and raise if a kernel gave up on a bounded wait."""
    check(load().ra_device_status(_stream(stream)))


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)
