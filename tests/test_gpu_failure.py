"""Failure detection without a GPU fault: every on-chip wait of the bf16
kernel has a time budget. With the test hook RA_TEST_STALL=1 each CTA first
waits on an mbarrier that nothing ever completes; the wait must give up after
the budget (RA_WAIT_BUDGET_NS), the kernel must let its in-flight copies and
MMAs finish, free its TMEM and return, and ra_device_status must report
RA_ERR_TIMEOUT. The same process must then compute correctly again."""
import math

import numpy as np
import pytest
import torch

import oracle
from blockwise_attention_online_gb300 import RaError, _lib, device_status, ring_attention
from _util import assert_bf16, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs():
    g = torch.Generator(device="cpu").manual_seed(41)
    q = torch.randn(1, 2, 640, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 2, 640, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 2, 640, 128, generator=g).to(torch.bfloat16)
    return q, k, v


def test_stalled_wait_times_out_and_the_context_survives(monkeypatch):
    q, k, v = _inputs()
    qd, kc, vc = q.to(DEV), [k.to(DEV)], [v.to(DEV)]
    device_status()                                  # start from a clean status word
    monkeypatch.setenv("RA_WAIT_BUDGET_NS", str(20_000_000))   # 20 ms
    monkeypatch.setenv("RA_TEST_STALL", "1")
    ring_attention(qd, kc, vc, causal=True)          # enqueues fine ...
    with pytest.raises(RaError) as err:              # ... and reports the timeout
        device_status()
    assert err.value.status == _lib.RA_ERR_TIMEOUT
    assert "gave up waiting" in str(err.value)
    device_status()                                  # the read cleared the flag
    monkeypatch.delenv("RA_TEST_STALL")
    monkeypatch.delenv("RA_WAIT_BUDGET_NS")
    O, m, l = ring_attention(qd, kc, vc, causal=True)
    device_status()
    pos = np.arange(640)
    ref = oracle.full_attention(f64(q), f64(k), f64(v), pos, pos, True, 1 / math.sqrt(128))
    assert_bf16(O, m, l, *ref, what="after a timed-out launch")
