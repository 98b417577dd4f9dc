"""Seeded synthetic inputs for the ring-attention forward pass.

This module holds no attention arithmetic. It only names the workloads and
draws their Q, K, V tensors, so that the CUDA path and the fp64 checker can be
fed the very same values. Tensors come back in GLOBAL sequence order with
shape [B, H, S, D]; splitting into per-device chunks (contiguous, zigzag,
striped) is done by ``layouts``.

Recipe: fp32 ``torch.randn`` on a generator seeded with ``seed``, drawn in the
order Q, K, V; Q and K are multiplied by ``qk_gain`` (a power of two, so the
product is exact) and all three are then rounded to the working dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "f32" or "bf16": the type the inputs are stored in
    B: int
    Hq: int
    Hkv: int
    S: int              # queries == keys
    D: int
    causal: bool
    n_chunks: int
    layout: str         # "contiguous" | "zigzag" | "striped"
    seed: int
    qk_gain: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def flops(self) -> float:
        """Algorithmic FLOPs of one forward: 4*B*Hq*Sq*Sk*D (QK^T and PV,
        two flops per multiply-add); halved for causal masks."""
        f = 4.0 * self.B * self.Hq * self.S * self.S * self.D
        return f / 2 if self.causal else f


WORKLOADS = {
    # fp32, one head, 256 x 256, head_dim 64, 4 contiguous chunks of 64.
    "fp32_256": Workload("fp32_256", "f32", 1, 1, 1, 256, 64, False, 4,
                         "contiguous", 0),
    # bf16, 8 heads, 8192 tokens, head_dim 128, non-causal, 8 chunks of 1024.
    "bf16_8k": Workload("bf16_8k", "bf16", 1, 8, 8, 8192, 128, False, 8,
                        "contiguous", 2),
    # bf16, 32 heads, 32768 tokens, causal, 8 contiguous chunks of 4096.
    "bf16_32k_causal": Workload("bf16_32k_causal", "bf16", 1, 32, 32, 32768,
                                128, True, 8, "contiguous", 3),
    # bf16, 32 query heads over 8 K/V heads, 131072 tokens, causal,
    # 16 zigzag chunks of 8192 (also run contiguous and striped).
    "bf16_128k_gqa_causal": Workload("bf16_128k_gqa_causal", "bf16", 1, 32, 8,
                                     131072, 128, True, 16, "zigzag", 4),
    # bf16, 8 heads, 1M tokens, causal, 8 chunks of 131072, Q/K scaled by 4 so
    # that scaled logits reach about +-60.
    "bf16_1m_causal": Workload("bf16_1m_causal", "bf16", 1, 8, 8, 1048576, 128,
                               True, 8, "contiguous", 5, 4.0),
}


def make_generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_qkv(w: Workload, device="cpu", S: int | None = None, seed: int | None = None):
    """Draw (q, k, v) for workload ``w`` on ``device`` in global order.

    ``S`` overrides the sequence length (for reduced-size cases of the same
    workload), ``seed`` the seed. The draw happens on ``device`` with a
    generator of that device type.
    """
    S = w.S if S is None else S
    seed = w.seed if seed is None else seed
    g = make_generator(seed, device)
    shp_q = (w.B, w.Hq, S, w.D)
    shp_kv = (w.B, w.Hkv, S, w.D)
    out = []
    for shp, gain in ((shp_q, w.qk_gain), (shp_kv, w.qk_gain), (shp_kv, 1.0)):
        t = torch.randn(shp, generator=g, dtype=torch.float32, device=device)
        if gain != 1.0:
            t.mul_(gain)
        out.append(t.to(w.torch_dtype))
        del t
    return tuple(out)


def packed_documents(S: int, seed: int, mean_len: int, min_len: int = 1) -> list[int]:
    """Boundaries b_0 = 0 < b_1 < ... < b_n = S of packed documents whose
    lengths are drawn log-uniformly in [min_len, 4 * mean_len) with ``seed``
    (many short documents, a few long ones; the last is cut at S)."""
    rng = np.random.default_rng(seed)
    hi = max(min_len + 1, 4 * mean_len)
    b = [0]
    while b[-1] < S:
        n = int(np.exp(rng.uniform(np.log(min_len), np.log(hi))))
        b.append(min(S, b[-1] + max(min_len, n)))
    return b


def scalar_two_shards():
    """The two-shard scalar case: one query, shard A holds a key giving score 0
    with value 0, shard B a key giving score 10 with value 1 (head_dim 1,
    scale 1). Returns q [1,1,1,1], k chunks and v chunks (each [1,1,1,1])."""
    q = torch.ones(1, 1, 1, 1, dtype=torch.float32)
    ka = torch.zeros(1, 1, 1, 1, dtype=torch.float32)
    kb = torch.full((1, 1, 1, 1), 10.0, dtype=torch.float32)
    va = torch.zeros(1, 1, 1, 1, dtype=torch.float32)
    vb = torch.ones(1, 1, 1, 1, dtype=torch.float32)
    return q, [ka, kb], [va, vb]
