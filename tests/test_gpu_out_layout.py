"""The bf16 forward writes O through any output layout the header allows
(strides in multiples of 8 elements): a head-interleaved view ([B, S, H, D]
memory read as [B, H, S, D]) and rows padded to a wider pitch give exactly
the contiguous result, and nothing outside the view is written. head_dim 128
(where O leaves through TMA stores of 32-row boxes) and 96, sequence lengths
that are not multiples of 32 or 256, causal and not; the contiguous result
itself is checked against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_attention_online_gb300 import device_status, ring_attention
from _util import assert_bf16, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(H, S, D, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    q, k, v = (torch.randn(1, H, S, D, generator=g).to(torch.bfloat16) for _ in range(3))
    return q, k, v


@pytest.mark.parametrize("S,D,causal", [(1000, 128, False), (1000, 128, True), (333, 96, True),
                                        (40, 128, False)])
def test_bf16_output_views(S, D, causal):
    H = 4
    q, k, v = _inputs(H, S, D, seed=S + D)
    lens = [S // 3, S // 3, S - 2 * (S // 3)]
    qd = q.to(DEV)
    kc = [x.contiguous() for x in torch.split(k.to(DEV), lens, dim=2)]
    vc = [x.contiguous() for x in torch.split(v.to(DEV), lens, dim=2)]
    scale = 1.0 / D ** 0.5

    O0, m0, l0 = ring_attention(qd, kc, vc, causal=causal)
    device_status()
    ref = oracle.full_attention(f64(q), f64(k), f64(v), np.arange(S), np.arange(S), causal, scale)
    assert_bf16(O0, m0, l0, *ref, what=f"contiguous S={S} D={D}")

    # head-interleaved: memory [1, S, H, D], viewed as [1, H, S, D]
    inter = torch.full((1, S, H, D), 7.0, device=DEV, dtype=torch.bfloat16)
    O1, _, _ = ring_attention(qd, kc, vc, causal=causal, out=inter.permute(0, 2, 1, 3))
    device_status()
    assert torch.equal(O1, O0)
    assert torch.equal(inter.permute(0, 2, 1, 3), O0)

    # rows padded to D + 64 elements; the padding must stay untouched
    pad = torch.full((1, H, S, D + 64), 7.0, device=DEV, dtype=torch.bfloat16)
    O2, _, _ = ring_attention(qd, kc, vc, causal=causal, out=pad[..., :D])
    device_status()
    assert torch.equal(O2, O0)
    assert torch.all(pad[..., D:] == 7.0)
