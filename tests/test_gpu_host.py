"""ra_ring_attention_host: the ring pass with every tensor in host memory.

The entry point copies the inputs in, runs the same kernel as
ra_ring_attention and copies O, m, l back, stream-ordered. Its results must be
those of the device entry point on the same inputs, bit for bit, and within
the oracle's tolerances; calls on two streams at once must not disturb each
other (each call has its own device copies).
"""
import numpy as np
import pytest
import torch

import oracle
from blockwise_attention_online_gb300 import layouts, ring_attention, ring_attention_host
from _util import assert_bf16, assert_f32, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, dtype, B, Hq, Hkv, S, D, kind, P):
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(B, Hq, S, D, generator=g).to(dtype)
    k = torch.randn(B, Hkv, S, D, generator=g).to(dtype)
    v = torch.randn(B, Hkv, S, D, generator=g).to(dtype)
    rs = layouts.rank_spans(kind, S, P)
    kc = [t.contiguous() for t in layouts.shard(k, kind, P)]
    vc = [t.contiguous() for t in layouts.shard(v, kind, P)]
    qs = torch.cat(layouts.shard(q, kind, P), dim=2).contiguous()
    segs = [(S // P, s) for s in rs]
    return q, k, v, qs, kc, vc, rs, segs


def _pinned(ts):
    return [t.pin_memory() for t in ts]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,S,D,kind,P,causal,out_dtype", [
    (torch.bfloat16, 1, 8, 2, 2048, 128, "zigzag", 4, True, None),
    (torch.bfloat16, 2, 4, 4, 1536, 64, "contiguous", 3, False, torch.float32),
    (torch.float32, 1, 2, 1, 384, 64, "striped", 4, True, None),
])
def test_host_entry_equals_device_entry(dtype, B, Hq, Hkv, S, D, kind, P, causal, out_dtype):
    q, k, v, qs, kc, vc, rs, segs = _case(7, dtype, B, Hq, Hkv, S, D, kind, P)
    hq = qs.pin_memory()
    hk, hv = _pinned(kc), _pinned(vc)
    stream = torch.cuda.Stream()
    O, m, l = ring_attention_host(hq, hk, hv, chunk_spans=rs, q_segments=segs, causal=causal,
                                  out_dtype=out_dtype, stream=stream)
    stream.synchronize()
    assert not O.is_cuda and O.dtype == (out_dtype or dtype)
    Od, md, ld = ring_attention(qs.to(DEV), [t.to(DEV) for t in kc], [t.to(DEV) for t in vc],
                                chunk_spans=rs, q_segments=segs, causal=causal,
                                out_dtype=out_dtype)
    torch.cuda.synchronize()
    # the same kernel and schedule: identical results
    assert torch.equal(O, Od.cpu()) and torch.equal(m, md.cpu()) and torch.equal(l, ld.cpu())
    # and the oracle agrees
    Og = layouts.to_global(O, kind, P)
    mg = layouts.to_global(m.unsqueeze(-1), kind, P).squeeze(-1)
    lg = layouts.to_global(l.unsqueeze(-1), kind, P).squeeze(-1)
    pos = np.arange(S)
    Hg = Hq // Hkv
    kr = f64(k).repeat(Hg, axis=1)
    vr = f64(v).repeat(Hg, axis=1)
    Oref, mref, lref = oracle.full_attention(f64(q), kr, vr, pos, pos, causal, D ** -0.5)
    if dtype == torch.float32:
        assert_f32(Og, mg, lg, Oref, mref, lref)
    else:
        assert_bf16(Og, mg, lg, Oref, mref, lref, what="host entry")


def test_two_streams_overlap_without_interference():
    """Alternate calls over two streams with different inputs (copies of one
    call overlap the other call's kernel); every result must equal the device
    entry point's."""
    cases = [_case(20 + i, torch.bfloat16, 1, 8, 8, 2048, 128, "contiguous", 2) for i in range(4)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    results = []
    for i, (q, k, v, qs, kc, vc, rs, segs) in enumerate(cases):
        hq = qs.pin_memory()
        hk, hv = _pinned(kc), _pinned(vc)
        out = ring_attention_host(hq, hk, hv, chunk_spans=rs, q_segments=segs, causal=True,
                                  stream=streams[i % 2])
        results.append((out, (hq, hk, hv)))   # keep the host inputs alive until the sync
    torch.cuda.synchronize()
    for (q, k, v, qs, kc, vc, rs, segs), ((O, m, l), _) in zip(cases, results):
        Od, md, ld = ring_attention(qs.to(DEV), [t.to(DEV) for t in kc], [t.to(DEV) for t in vc],
                                    chunk_spans=rs, q_segments=segs, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(O, Od.cpu()) and torch.equal(m, md.cpu()) and torch.equal(l, ld.cpu())


def _one_pinned_block(tensors, copy=True):
    sizes = [t.numel() * t.element_size() for t in tensors]
    buf = torch.empty(sum(sizes), dtype=torch.uint8, pin_memory=True)
    views, at = [], 0
    for t, n in zip(tensors, sizes):
        view = buf[at:at + n].view(t.dtype).view(t.shape)
        if copy:
            view.copy_(t)
        views.append(view)
        at += n
    return views


def test_host_buffers_in_one_block():
    """Q, the K chunks and the V chunks back to back in one pinned buffer, and
    O, m, l in another: the entry point merges copies of tensors adjacent on
    the host and on the device (ragged chunks of head_dim 96 leave padding
    between some device copies, and one chunk is empty), with results equal to
    the device entry point's."""
    S, D, Hq, Hkv = 1500, 96, 4, 2
    g = torch.Generator(device="cpu").manual_seed(31)
    q = torch.randn(1, Hq, S, D, generator=g).bfloat16()
    k = torch.randn(1, Hkv, S, D, generator=g).bfloat16()
    v = torch.randn(1, Hkv, S, D, generator=g).bfloat16()
    lens = [256, 300, 0, 128, 1, 431, 384]
    assert sum(lens) == S
    kc = [t.contiguous() for t in torch.split(k, lens, dim=2)]
    vc = [t.contiguous() for t in torch.split(v, lens, dim=2)]
    hq, *hkv = _one_pinned_block([q, *kc, *vc])
    O_like = torch.empty(1, Hq, S, D, dtype=torch.bfloat16)
    ml_like = torch.empty(1, Hq, S, dtype=torch.float32)
    ho, hm, hl = _one_pinned_block([O_like, ml_like, ml_like], copy=False)
    stream = torch.cuda.Stream()
    for causal in (False, True):
        O, m, l = ring_attention_host(hq, hkv[:len(lens)], hkv[len(lens):], causal=causal,
                                      out=ho, m=hm, l=hl, stream=stream)
        stream.synchronize()
        Od, md, ld = ring_attention(q.to(DEV), [t.to(DEV) for t in kc],
                                    [t.to(DEV) for t in vc], causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(O, Od.cpu()) and torch.equal(m, md.cpu()) and torch.equal(l, ld.cpu())
        pos = np.arange(S)
        Oref, mref, lref = oracle.full_attention(f64(q), f64(k).repeat(2, axis=1),
                                                 f64(v).repeat(2, axis=1), pos, pos, causal,
                                                 D ** -0.5)
        assert_bf16(O, m, l, Oref, mref, lref, what=f"one-block host buffers causal={causal}")
