"""ctypes view of the C ABI in include/ra.h (argument marshalling only).

The shared library is built in-tree (``_build/libra.so``). Loading fails loudly
when it is missing: there is no CPU fallback for any entry point.
"""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import POINTER, c_float, c_int32, c_int64, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libra.so")

RA_OK, RA_ERR_INVALID, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_TIMEOUT = range(5)
RA_F32, RA_BF16 = 0, 1
RA_MAX_SPANS = 4
STATUS_NAMES = {0: "RA_OK", 1: "RA_ERR_INVALID", 2: "RA_ERR_UNSUPPORTED",
                3: "RA_ERR_CUDA", 4: "RA_ERR_TIMEOUT"}

# every symbol include/ra.h declares
EXPORTED = ("ra_chunk_stats", "ra_merge_stats", "ra_ring_attention",
            "ra_ring_attention_noalloc", "ra_ring_attention_host", "ra_ring_attention_bwd",
            "ra_merge_lse", "ra_stats_to_lse", "ra_segment_work", "ra_device_status",
            "ra_last_error", "ra_version")


class Span(ctypes.Structure):
    _fields_ = [("len", c_int64), ("pos0", c_int64), ("step", c_int64)]


class Positions(ctypes.Structure):
    _fields_ = [("nspan", c_int32), ("reserved", c_int32), ("span", Span * RA_MAX_SPANS)]


class Strides(ctypes.Structure):
    _fields_ = [("batch", c_int64), ("head", c_int64), ("row", c_int64)]


class KvChunk(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("len", c_int64),
                ("k_strides", Strides), ("v_strides", Strides), ("pos", Positions)]


class KvGrad(ctypes.Structure):
    _fields_ = [("dk", c_void_p), ("dv", c_void_p)]


class QSegment(ctypes.Structure):
    _fields_ = [("len", c_int64), ("pos", Positions)]


class Problem(ctypes.Structure):
    _fields_ = [("B", c_int64), ("Hq", c_int64), ("Hkv", c_int64), ("D", c_int64),
                ("Sq", c_int64), ("dtype", c_int32), ("causal", c_int32),
                ("scale", c_float), ("o_fp32", c_int32),
                ("q_strides", Strides), ("o_strides", Strides),
                ("doc_bounds", c_void_p), ("n_docs", c_int32), ("reserved_docs", c_int32)]


class RaError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


_lib = None
_lock = threading.Lock()


def load():
    """Load libra.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m blockwise_attention_online_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(LIB_PATH)
        P = POINTER
        lib.ra_chunk_stats.argtypes = [P(Problem), c_void_p, P(QSegment), c_int32, P(KvChunk),
                                       c_void_p, c_void_p, c_void_p, c_void_p]
        lib.ra_merge_stats.argtypes = [c_int64, c_int64, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p, c_void_p]
        lib.ra_ring_attention.argtypes = [P(Problem), c_void_p, P(QSegment), c_int32,
                                          P(KvChunk), c_int32, c_void_p, c_void_p, c_void_p,
                                          c_void_p]
        lib.ra_ring_attention_noalloc.argtypes = lib.ra_ring_attention.argtypes
        lib.ra_ring_attention_host.argtypes = lib.ra_ring_attention.argtypes
        lib.ra_ring_attention_bwd.argtypes = [P(Problem), c_void_p, P(QSegment), c_int32,
                                              P(KvChunk), c_int32, c_void_p, c_void_p, c_void_p,
                                              c_void_p, c_void_p, P(KvGrad), c_void_p]
        lib.ra_merge_lse.argtypes = [c_int64, c_int64, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p]
        lib.ra_stats_to_lse.argtypes = [c_int64, c_void_p, c_void_p, c_void_p, c_void_p]
        lib.ra_segment_work.argtypes = [P(Problem), P(QSegment), c_int32, P(KvChunk), c_int32,
                                        c_void_p, c_void_p]
        lib.ra_device_status.argtypes = [c_void_p]
        lib.ra_last_error.restype = ctypes.c_char_p
        lib.ra_last_error.argtypes = []
        lib.ra_version.restype = c_int32
        lib.ra_version.argtypes = []
        for name in ("ra_chunk_stats", "ra_merge_stats", "ra_ring_attention",
                     "ra_ring_attention_noalloc", "ra_ring_attention_host",
                     "ra_ring_attention_bwd", "ra_merge_lse", "ra_stats_to_lse",
                     "ra_segment_work", "ra_device_status"):
            getattr(lib, name).restype = c_int32
        _lib = lib
        return lib


def check(status):
    if status != RA_OK:
        msg = load().ra_last_error().decode(errors="replace")
        raise RaError(status, msg)


def positions(spans):
    """Positions struct from a list of (len, pos0, step) tuples."""
    spans = list(spans)
    if not 1 <= len(spans) <= RA_MAX_SPANS:
        raise ValueError(f"need 1..{RA_MAX_SPANS} spans, got {len(spans)}")
    p = Positions()
    p.nspan = len(spans)
    p.reserved = 0
    for i, (n, p0, st) in enumerate(spans):
        p.span[i] = Span(int(n), int(p0), int(st))
    return p
