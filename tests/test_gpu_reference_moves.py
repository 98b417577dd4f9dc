"""Rows whose running maximum jumps inside a 128-key tile.

The bf16 kernel's one-pass softmax exponentiates each 32-column chunk of a
score tile against the row's reference maximum and moves the reference only
when a chunk's maximum exceeds it by a wide margin (the P chunks already
written for that tile, the row sums and O are rescaled first); the two-pass
form rescales O whenever the row max grows past a small margin. These
inputs make that happen at every chunk position of a tile and on many
tiles in a row (one key dimension carries spikes whose height grows by tens
of nats from one tile to the next), while other rows see dips instead (no
move at all), under both forms. The result must still be the exact softmax: the oracle's
definition, within the bf16 tolerances ("Online softmax": the rescale
factor exp(m_old - m_new) applied to the running numerator and denominator).
"""
import numpy as np
import pytest
import torch

import oracle
from blockwise_attention_online_gb300 import device_status, ring_attention
from _util import assert_bf16, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _spiky(seed, Hq, S, D):
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(1, Hq, S, D, generator=g) * 0.5
    k = torch.randn(1, Hq, S, D, generator=g) * 0.5
    v = torch.randn(1, Hq, S, D, generator=g)
    scale = D ** -0.5
    # dimension 0: the query's sign decides whether a row sees the spikes
    sign = torch.where(torch.rand(1, Hq, S, generator=g) < 0.5, -1.0, 1.0)
    q[..., 0] = 4.0 * sign
    rng = np.random.default_rng(seed)
    height = 0.0
    for t in range(S // 128):
        # one spike per tile, in a varying 32-column chunk, 30-45 nats higher
        # than the last one (more than the 32-bit-exponent slack of 22 nats)
        height += float(rng.uniform(30.0, 45.0))
        col = 128 * t + int(rng.integers(0, 128))
        k[0, :, col, 0] = height / (4.0 * scale)
    return q.bfloat16(), k.bfloat16(), v.bfloat16(), scale


# docs=[0, S]: one document over the whole sequence masks nothing but, without
# a causal mask, selects the kernel's one-pass softmax (the form used with
# packed documents); otherwise the two-pass form runs
FORMS = [None, "whole"]


def _docs(form, S):
    return None if form is None else [0, S]


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("causal", [False, True])
def test_reference_moves_inside_tiles(causal, form):
    Hq, S, D = 2, 1280, 64
    q, k, v, scale = _spiky(41, Hq, S, D)
    kc = [t.contiguous().to(DEV) for t in torch.split(k, 256, dim=2)]
    vc = [t.contiguous().to(DEV) for t in torch.split(v, 256, dim=2)]
    O, m, l = ring_attention(q.to(DEV), kc, vc, causal=causal, docs=_docs(form, S))
    device_status()
    pos = np.arange(S)
    Oref, mref, lref = oracle.full_attention(f64(q), f64(k), f64(v), pos, pos, causal, scale)
    assert np.nanmax(np.abs(mref[np.isfinite(mref)])) > 200.0   # the spikes really are tall
    assert_bf16(O, m, l, Oref, mref, lref, what=f"spiky rows causal={causal} form={form}")


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("causal", [True, False])
def test_reference_moves_with_fp32_output_and_split_units(form, causal):
    """The same rows with many query tiles per head (units split across CTAs,
    partial results merged) and fp32 O."""
    Hq, S, D = 8, 4096, 128
    q, k, v, scale = _spiky(42, Hq, S, D)
    kc = [t.contiguous().to(DEV) for t in torch.split(k, 1024, dim=2)]
    vc = [t.contiguous().to(DEV) for t in torch.split(v, 1024, dim=2)]
    O, m, l = ring_attention(q.to(DEV), kc, vc, causal=causal, out_dtype=torch.float32,
                             docs=_docs(form, S))
    device_status()
    pos = np.arange(S)
    Oref, mref, lref = oracle.full_attention(f64(q), f64(k), f64(v), pos, pos, causal, scale)
    assert_bf16(O, m, l, Oref, mref, lref, what=f"spiky rows fp32 O causal={causal}")
