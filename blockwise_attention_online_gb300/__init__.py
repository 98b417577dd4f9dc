"""GB300-native chunked (ring) attention forward: a C-ABI CUDA library
(``_build/libra.so``, sources in ``csrc/``, header ``include/ra.h``) and a thin
torch binding. The binding loads the library on first use and raises if it
has not been built; there is no CPU fallback.
"""
from .api import (chunk_stats, default_scale, device_status, merge_lse, merge_stats,
                  ring_attention, ring_attention_bwd, ring_attention_host, segment_work,
                  stats_to_lse)
from ._lib import RaError

__all__ = ["chunk_stats", "default_scale", "device_status", "merge_lse", "merge_stats",
           "stats_to_lse",
           "ring_attention", "ring_attention_bwd", "ring_attention_host", "segment_work",
           "RaError"]
