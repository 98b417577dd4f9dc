"""fp64 CPU oracle for ring attention's chunked forward pass and its backward.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU legs of bench.py, never by the library. See ``oracle.attention``.
"""
from .attention import (NEG_INF, attention_rows, chunk_stats, document_of, full_attention,
                        merge_stats, normalize, ring_attention, ring_order,
                        unmasked_pairs)
from .backward import attention_backward, gradient_rounding_bounds, ring_attention_backward
from .lse import merge_lse, stats_to_lse
from . import layouts

__all__ = ["NEG_INF", "attention_rows", "chunk_stats", "document_of", "full_attention",
           "merge_stats", "normalize", "ring_attention", "ring_order",
           "unmasked_pairs", "layouts", "attention_backward", "gradient_rounding_bounds",
           "ring_attention_backward",
           "merge_lse", "stats_to_lse"]
