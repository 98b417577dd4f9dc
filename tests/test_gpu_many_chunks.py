"""Problems with more chunks or spans than the launch plan itself holds (32
chunks, 64 spans): their chunk tables (tensor maps, spans) live in device
memory. The exercise asks that the chunked pass equal ordinary attention for
every way of splitting the keys, down to chunks of one key (exercise page
"systems-distributed-ring-attention-online-softmax", task statement); a ring
of 64 devices needs 64 chunks.

Every case is compared with the fp64 oracle at the bf16 tolerances
(O max-abs 1e-2, m and l relative 1e-3); the backward at the normwise bound
of its own tests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from blockwise_attention_online_gb300 import device_status, ring_attention, ring_attention_bwd
from _util import assert_bf16, f64, layout_run

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed, B, Hq, Hkv, S, D):
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(B, Hq, S, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    return q, k, v


def _ref(q, k, v, causal, D):
    pos = np.arange(k.shape[2])
    return oracle.full_attention(f64(q), f64(k), f64(v), np.arange(q.shape[2]), pos, causal,
                                 1 / math.sqrt(D))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("out_dtype", [None, torch.float32])
def test_size1_chunks_ring(causal, out_dtype):
    """256 chunks of one key each, walked in ring order by 256 one-row query
    segments (each segment plays one device of a 256-device ring)."""
    S, D = 256, 128
    q, k, v = _inputs(101, 1, 2, 1, S, D)
    kc = [t.contiguous() for t in torch.split(k.to(DEV), 1, dim=2)]
    vc = [t.contiguous() for t in torch.split(v.to(DEV), 1, dim=2)]
    spans = [[(1, i, 1)] for i in range(S)]
    segs = [(1, [(1, i, 1)]) for i in range(S)]
    O, m, l = ring_attention(q.to(DEV), kc, vc, chunk_spans=spans, q_segments=segs,
                             causal=causal, out_dtype=out_dtype)
    device_status()
    assert_bf16(O, m, l, *_ref(q, k, v, causal, D), what="256 size-1 chunks")


@pytest.mark.parametrize("kind", ["contiguous", "zigzag", "striped"])
def test_64_device_ring(kind):
    """A 64-device ring: 64 chunks (zigzag: 128 spans) and 64 query segments,
    causal with global positions, grouped heads."""
    S, D = 4096, 128
    q, k, v = _inputs(102, 1, 4, 2, S, D)
    O, m, l = layout_run(q.to(DEV), k.to(DEV), v.to(DEV), 64, kind, True)
    device_status()
    assert_bf16(O, m, l, *_ref(q, k, v, True, D), what=f"64-device {kind} ring")


def test_many_ragged_chunks_index_order():
    """40 chunks of uneven lengths (some empty) walked in index order by one
    segment, head_dim 96, every unit split across CTAs."""
    S, D = 1500, 96
    q, k, v = _inputs(103, 1, 2, 2, S, D)
    rng = np.random.default_rng(5)
    cuts = np.sort(rng.choice(np.arange(1, S), size=39, replace=False))
    lens = np.diff(np.concatenate([[0], cuts, [S]])).tolist()
    lens[3] = lens[3] + lens[4]
    lens[4] = 0                                         # an empty chunk
    kc = [t.contiguous() for t in torch.split(k.to(DEV), lens, dim=2)]
    vc = [t.contiguous() for t in torch.split(v.to(DEV), lens, dim=2)]
    for causal in (False, True):
        O, m, l = ring_attention(q.to(DEV), kc, vc, causal=causal)
        device_status()
        assert_bf16(O, m, l, *_ref(q, k, v, causal, D), what=f"40 ragged chunks causal={causal}")


def test_backward_with_many_chunks():
    """The backward pass over 48 chunks (zigzag layout: 96 spans)."""
    from test_gpu_bwd import _check, _layout_bwd
    S, D = 1536, 128
    g = torch.Generator(device="cpu").manual_seed(104)
    q = torch.randn(1, 4, S, D, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 2, S, D, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 2, S, D, generator=g).to(torch.bfloat16)
    do = torch.randn(1, 4, S, D, generator=g).to(torch.bfloat16)
    dq, dk, dv = _layout_bwd(q, k, v, do, "zigzag", 16 * 3, True)
    pos = np.arange(S)
    rq, rk, rv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), pos, pos, True,
                                           D ** -0.5)
    _check("dq", dq, rq)
    _check("dk", dk, rk)
    _check("dv", dv, rv)
