"""Full-size workloads, in the launch configuration bench.py times, checked on
sampled rows against the fp64 oracle (each sampled row exact against all of
its visible keys) and, for every row, through properties that hold at any
size: no NaN/Inf, and agreement with a one-chunk run of the same problem
(chunk invariance, exercise task statement)."""
import numpy as np
import pytest
import torch

from blockwise_attention_online_gb300 import device_status, layouts, ring_attention, workloads
from _util import assert_bf16, f64, layout_run, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _global_inputs(name):
    w = workloads.WORKLOADS[name]
    q, k, v = workloads.make_qkv(w, device=DEV)
    return w, q, k, v


def _check_sampled(w, q, k, v, O, m, l, boundaries, heads, n_random=48):
    rows = sample_rows(w.S, boundaries, n_random)
    Or, mr, lr = oracle_rows(q, k, v, w.causal, w.scale, heads, rows)
    idx = torch.tensor(rows)
    for j, h in enumerate(heads):
        assert_bf16(O[0, h].index_select(0, idx.to(O.device)), m[0, h].index_select(0, idx.to(m.device)),
                    l[0, h].index_select(0, idx.to(l.device)), Or[j], mr[j], lr[j],
                    what=f"{w.name} head {h}")


def _invariance(O, m, l, O1, m1, l1):
    assert torch.isfinite(O.float()).all() and torch.isfinite(l).all()
    # two results, each within 1e-2 of the exact one
    assert (O.float() - O1.float()).abs().max().item() <= 2e-2
    rel = ((m - m1).abs() / m1.abs().clamp_min(1)).max().item()
    assert rel <= 1e-3
    assert ((l - l1).abs() / l1).max().item() <= 1e-3


def test_bf16_32k_causal_8_chunks():
    w, q, k, v = _global_inputs("bf16_32k_causal")
    O, m, l = layout_run(q, k, v, w.n_chunks, "contiguous", True)
    device_status()
    bnd = [i * (w.S // w.n_chunks) for i in range(1, w.n_chunks)]
    _check_sampled(w, q, k, v, O, m, l, bnd, heads=[0, 13, 31])
    O1, m1, l1 = ring_attention(q, [k], [v], causal=True)
    device_status()
    _invariance(O, m, l, O1, m1, l1)


@pytest.mark.parametrize("kind", ["zigzag", "contiguous", "striped"])
def test_bf16_128k_gqa_layouts(kind):
    """GQA 4:1, 131072 tokens, causal, 16 chunks of 8192; zigzag chunks are an
    early and a late 4096 block. Every layout must give the same attention."""
    w, q, k, v = _global_inputs("bf16_128k_gqa_causal")
    O, m, l = layout_run(q, k, v, w.n_chunks, kind, True)
    device_status()
    half = w.S // (2 * w.n_chunks)
    bnd = [i * half for i in range(1, 2 * w.n_chunks)]
    _check_sampled(w, q, k, v, O, m, l, bnd, heads=[0, 5, 30], n_random=32)
    if kind == "zigzag":
        O1, m1, l1 = ring_attention(q, [k], [v], causal=True)
        device_status()
        _invariance(O, m, l, O1, m1, l1)


def test_bf16_1m_causal_wide_logits():
    """1M tokens, causal, 8 chunks of 131072, Q and K scaled by 4 so scaled
    logits span about +-60: stresses the max-rescale merge. Attention is then
    dominated by one key per row, so |O| reaches 4 and more, where a bf16 O's
    own rounding alone exceeds 1e-2: the 1e-2 bound is checked on an fp32 O,
    the bf16 O against 1e-2 plus its rounding."""
    w, q, k, v = _global_inputs("bf16_1m_causal")
    bnd = [i * (w.S // w.n_chunks) for i in range(1, w.n_chunks)]
    O32, m32, l32 = layout_run(q, k, v, w.n_chunks, "contiguous", True, out_dtype=torch.float32)
    device_status()
    assert m32.abs().max().item() > 40.0        # the logits really are wide
    _check_sampled(w, q, k, v, O32, m32, l32, bnd, heads=[0, 7], n_random=24)
    O, m, l = layout_run(q, k, v, w.n_chunks, "contiguous", True)
    device_status()
    assert torch.equal(m, m32) and torch.equal(l, l32)
    assert torch.equal(O, O32.to(torch.bfloat16))
    del O
    # chunk invariance at full size, on fp32 outputs (two bf16 outputs may
    # differ by an ulp, 0.031 at |O| >= 4)
    O1, m1, l1 = ring_attention(q, [k], [v], causal=True, out_dtype=torch.float32)
    device_status()
    _invariance(O32, m32, l32, O1, m1, l1)
