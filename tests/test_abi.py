"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects invalid arguments before anything is launched.
Also the host-only bookkeeping (layout spans, per-segment work) against the
oracle, bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from oracle import layouts as olay
from blockwise_attention_online_gb300 import _lib, layouts, segment_work

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_symbols():
    with open(os.path.join(ROOT, "include", "ra.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(ra_[a-z_]+)\s*\(", text)))


def test_library_exports_every_header_symbol():
    lib = _lib.load()
    declared = _header_symbols()
    assert set(declared) == set(_lib.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.ra_version() == 101


def _problem(**kw):
    p = _lib.Problem()
    p.B, p.Hq, p.Hkv, p.D, p.Sq = kw.get("B", 1), kw.get("Hq", 2), kw.get("Hkv", 1), \
        kw.get("D", 128), kw.get("Sq", 256)
    p.dtype = kw.get("dtype", _lib.RA_BF16)
    p.causal = kw.get("causal", 0)
    p.scale = kw.get("scale", 0.0)
    p.o_fp32 = kw.get("o_fp32", 0)
    D, Sq, Hq = p.D, p.Sq, p.Hq
    p.q_strides = _lib.Strides(Hq * Sq * D, Sq * D, D)
    p.o_strides = _lib.Strides(Hq * Sq * D, Sq * D, D)
    return p


def _segs(spec):
    arr = (_lib.QSegment * len(spec))()
    for i, (n, spans) in enumerate(spec):
        arr[i].len = n
        arr[i].pos = _lib.positions(spans)
    return arr


def _chunks(spec, ptr=4096, D=128, Hkv=1):
    arr = (_lib.KvChunk * len(spec))()
    for i, (n, spans) in enumerate(spec):
        arr[i].k = ptr
        arr[i].v = ptr
        arr[i].len = n
        st = _lib.Strides(Hkv * n * D, n * D, D)
        arr[i].k_strides = st
        arr[i].v_strides = st
        arr[i].pos = _lib.positions(spans)
    return arr


def _call(p, segs, nsegs, chunks, nchunks, q=4096, o=4096, m=4096, l=4096):
    lib = _lib.load()
    return lib.ra_ring_attention(ctypes.byref(p), q, segs, nsegs, chunks, nchunks, o, m, l, None)


GOOD_SEGS = [(256, [(256, 0, 1)])]
GOOD_CHUNKS = [(128, [(128, 0, 1)]), (128, [(128, 128, 1)])]


@pytest.mark.parametrize("bad", [
    dict(Hq=3, Hkv=2),                 # Hq not a multiple of Hkv
    dict(D=80),                        # bf16 head_dim outside {64, 96, 128}
    dict(dtype=7),
    dict(causal=2),
    dict(o_fp32=2),
    dict(scale=float("nan")),
    dict(B=0),
])
def test_invalid_problem_rejected(bad):
    p = _problem(**bad)
    st = _call(p, _segs(GOOD_SEGS), 1, _chunks(GOOD_CHUNKS), 2)
    assert st in (_lib.RA_ERR_INVALID, _lib.RA_ERR_UNSUPPORTED)
    assert _lib.load().ra_last_error().decode()


def test_invalid_descriptors_rejected():
    p = _problem()
    lib = _lib.load()
    # segment lengths must add up to Sq
    assert _call(p, _segs([(200, [(200, 0, 1)])]), 1, _chunks(GOOD_CHUNKS), 2) == _lib.RA_ERR_INVALID
    # span lengths must add up to the segment's length
    assert _call(p, _segs([(256, [(255, 0, 1)])]), 1, _chunks(GOOD_CHUNKS), 2) == _lib.RA_ERR_INVALID
    # step must be >= 1
    assert _call(p, _segs([(256, [(256, 0, 0)])]), 1, _chunks(GOOD_CHUNKS), 2) == _lib.RA_ERR_INVALID
    # chunk spans must cover the chunk
    assert _call(p, _segs(GOOD_SEGS), 1, _chunks([(128, [(127, 0, 1)])]), 1) == _lib.RA_ERR_INVALID
    # positions must stay below 2^31 - 1
    assert _call(p, _segs([(256, [(256, 2**31 - 100, 1)])]), 1,
                 _chunks(GOOD_CHUNKS), 2) == _lib.RA_ERR_UNSUPPORTED
    # misaligned pointer for the TMA path
    assert _call(p, _segs(GOOD_SEGS), 1, _chunks(GOOD_CHUNKS, ptr=4098), 2) == _lib.RA_ERR_INVALID
    assert _call(p, _segs(GOOD_SEGS), 1, _chunks(GOOD_CHUNKS), 2, q=4100) == _lib.RA_ERR_INVALID
    # too many chunks for the bf16 path (its device-resident tables hold 4096)
    many = [(1, [(1, i, 1)]) for i in range(4097)]
    p2 = _problem(Sq=4097)
    assert _call(p2, _segs([(4097, [(4097, 0, 1)])]), 1, _chunks(many), 4097) == \
        _lib.RA_ERR_UNSUPPORTED
    # NULL outputs
    assert _call(p, _segs(GOOD_SEGS), 1, _chunks(GOOD_CHUNKS), 2, o=None) == _lib.RA_ERR_INVALID
    assert lib.ra_merge_stats(4, 0, 1, 1, 1, 1, 1, 1, None) == _lib.RA_ERR_INVALID
    assert lib.ra_merge_stats(-1, 8, 1, 1, 1, 1, 1, 1, None) == _lib.RA_ERR_INVALID
    assert lib.ra_merge_stats(4, 8, None, 16, 16, 16, 16, 16, None) == _lib.RA_ERR_INVALID
    # an empty problem is a valid no-op
    assert _call(_problem(Sq=0), _segs([(0, [(0, 0, 1)])]), 1, _chunks(GOOD_CHUNKS), 2) == _lib.RA_OK
    assert lib.ra_merge_stats(0, 8, None, None, None, None, None, None, None) == _lib.RA_OK


@pytest.mark.parametrize("kind", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("n,P", [(64, 4), (1024, 8), (96, 2)])
def test_layout_spans_match_oracle_positions(kind, n, P):
    got = [layouts.span_positions(s).numpy() for s in layouts.rank_spans(kind, n, P)]
    want = olay.positions(kind, n, P)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)
    x = torch.arange(n).view(1, 1, n, 1).float()
    sh = torch.cat(layouts.shard(x, kind, P), dim=2)
    assert torch.equal(layouts.to_global(sh, kind, P), x)


@pytest.mark.parametrize("kind", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("causal", [False, True])
def test_segment_work_is_exact(kind, causal):
    """Visible (query, key) pairs per virtual rank: bit-exact against the
    oracle's count; the scheduled tile products cover them."""
    n, P = 4096, 8
    rs = layouts.rank_spans(kind, n, P)
    segs = [(n // P, s) for s in rs]
    pairs, tiles = segment_work(1, 4, 4, 128, segs, [n // P] * P, rs, causal)
    allk = np.arange(n)
    want = [oracle.unmasked_pairs(p, allk, causal) for p in olay.positions(kind, n, P)]
    assert pairs == want
    assert all(t * 128 * 128 >= pr for t, pr in zip(tiles, pairs))
    if causal and kind == "zigzag":
        assert max(pairs) == min(pairs)


@pytest.mark.parametrize("kind", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("causal", [False, True])
def test_segment_work_with_documents_is_exact(kind, causal):
    """Packed documents: visible pairs per virtual rank bit-exact against the
    oracle's count; the scheduled tiles cover them and never exceed the
    unpacked schedule."""
    n, P = 4096, 8
    docs = [0, 1, 700, 701, 2048, 2100, 4000, 4096]
    rs = layouts.rank_spans(kind, n, P)
    segs = [(n // P, s) for s in rs]
    pairs, tiles = segment_work(1, 4, 4, 128, segs, [n // P] * P, rs, causal, docs=docs)
    _, tiles_plain = segment_work(1, 4, 4, 128, segs, [n // P] * P, rs, causal)
    allk = np.arange(n)
    want = [oracle.unmasked_pairs(p, allk, causal, docs) for p in olay.positions(kind, n, P)]
    assert pairs == want
    assert all(t * 128 * 128 >= pr for t, pr in zip(tiles, pairs))
    assert all(a <= b for a, b in zip(tiles, tiles_plain))
    if kind == "contiguous":
        assert sum(tiles) < sum(tiles_plain)
    with pytest.raises(ValueError):
        segment_work(1, 4, 4, 128, segs, [n // P] * P, rs, causal, docs=[0])
    # the most documents a call takes: 512 of 8 positions each
    many = list(range(0, n + 1, 8))
    assert len(many) - 1 == 512
    pairs512, _ = segment_work(1, 4, 4, 128, segs, [n // P] * P, rs, causal, docs=many)
    assert sum(pairs512) == (512 * (8 * 9 // 2) if causal else 512 * 64)
    # keys outside the documents are rejected, as by the launches
    with pytest.raises(_lib.RaError):
        segment_work(1, 4, 4, 128, segs, [n // P] * P, rs, causal, docs=docs[:-1] + [4095])


def test_documents_rejected():
    lib = _lib.load()

    def call(bounds, n_docs=None, reserved=0, segs=GOOD_SEGS, chunks=GOOD_CHUNKS):
        p = _problem()
        arr = (ctypes.c_int64 * max(1, len(bounds)))(*bounds)
        p.doc_bounds = ctypes.cast(arr, ctypes.c_void_p) if bounds else None
        p.n_docs = len(bounds) - 1 if n_docs is None else n_docs
        p.reserved_docs = reserved
        return _call(p, _segs(segs), len(segs), _chunks(chunks), len(chunks))

    assert call([0, 100, 100, 256]) == _lib.RA_ERR_INVALID      # not strictly increasing
    assert call([0, 200, 100, 256]) == _lib.RA_ERR_INVALID
    assert call([0, 255]) == _lib.RA_ERR_INVALID                 # position 255 outside
    assert call([1, 256]) == _lib.RA_ERR_INVALID                 # position 0 outside
    assert call([-1, 256]) == _lib.RA_ERR_INVALID
    assert call([0, 2**31]) == _lib.RA_ERR_INVALID
    assert call([], n_docs=1) == _lib.RA_ERR_INVALID             # NULL bounds
    assert call([0, 256], n_docs=-1) == _lib.RA_ERR_INVALID
    assert call(list(range(0, 514)), n_docs=513) == _lib.RA_ERR_INVALID   # > RA_MAX_DOCS
    assert call([0, 256], reserved=1) == _lib.RA_ERR_INVALID
    assert "document" in lib.ra_last_error().decode() or "reserved" in lib.ra_last_error().decode()
    # keys outside the documents are rejected too
    assert call([0, 256], chunks=[(128, [(128, 0, 1)]), (128, [(128, 200, 1)])]) == _lib.RA_ERR_INVALID


def _call_host(p, segs, nsegs, chunks, nchunks, q=4096, o=4096, m=4096, l=4096):
    lib = _lib.load()
    return lib.ra_ring_attention_host(ctypes.byref(p), q, segs, nsegs, chunks, nchunks,
                                      o, m, l, None)


def test_host_entry_rejects_before_touching_the_device():
    """ra_ring_attention_host validates everything, including that host
    tensors are dense, before it allocates or copies anything."""
    p = _problem()
    # the same descriptor checks as the device entry point
    assert _call_host(p, _segs([(200, [(200, 0, 1)])]), 1, _chunks(GOOD_CHUNKS), 2) == _lib.RA_ERR_INVALID
    assert _call_host(p, _segs(GOOD_SEGS), 1, _chunks(GOOD_CHUNKS), 2, o=None) == _lib.RA_ERR_INVALID
    # q padded between rows: not dense
    p2 = _problem()
    p2.q_strides = _lib.Strides(2 * 256 * 136, 256 * 136, 136)
    assert _call_host(p2, _segs(GOOD_SEGS), 1, _chunks(GOOD_CHUNKS), 2) == _lib.RA_ERR_INVALID
    assert "dense" in _lib.load().ra_last_error().decode()
    # O with a foreign head stride
    p3 = _problem()
    p3.o_strides = _lib.Strides(2 * 256 * 128, 512 * 128, 128)
    assert _call_host(p3, _segs(GOOD_SEGS), 1, _chunks(GOOD_CHUNKS), 2) == _lib.RA_ERR_INVALID
    # a chunk whose k rows are strided
    ch = _chunks(GOOD_CHUNKS)
    ch[1].k_strides = _lib.Strides(128 * 256, 128 * 256, 256)
    assert _call_host(p, _segs(GOOD_SEGS), 1, ch, 2) == _lib.RA_ERR_INVALID
    # an empty problem is a valid no-op
    assert _call_host(_problem(Sq=0), _segs([(0, [(0, 0, 1)])]), 1, _chunks(GOOD_CHUNKS), 2) == _lib.RA_OK


def _call_bwd(p, segs, nsegs, chunks, nchunks, grads, q=4096, o=4096, dout=4096, m=4096, l=4096,
              dq=4096):
    lib = _lib.load()
    return lib.ra_ring_attention_bwd(ctypes.byref(p), q, segs, nsegs, chunks, nchunks, o, dout,
                                     m, l, dq, grads, None)


def _grads(n, ptr=4096):
    g = (_lib.KvGrad * n)()
    for i in range(n):
        g[i].dk = ptr
        g[i].dv = ptr
    return g


def test_backward_entry_rejects_before_launch():
    p = _problem()
    segs, ch = _segs(GOOD_SEGS), _chunks(GOOD_CHUNKS)
    # head_dim outside {64, 96, 128}
    assert _call_bwd(_problem(D=80), segs, 1, _chunks(GOOD_CHUNKS, D=80), 2,
                     _grads(2)) == _lib.RA_ERR_UNSUPPORTED
    # fp32 inputs: the backward is bf16 only
    assert _call_bwd(_problem(dtype=_lib.RA_F32, D=64), segs, 1, _chunks(GOOD_CHUNKS, D=64), 2,
                     _grads(2)) == _lib.RA_ERR_UNSUPPORTED
    # gradient outputs missing
    assert _call_bwd(p, segs, 1, ch, 2, None) == _lib.RA_ERR_INVALID
    g = _grads(2)
    g[1].dv = None
    assert _call_bwd(p, segs, 1, ch, 2, g) == _lib.RA_ERR_INVALID
    # dout, dq or the statistics missing or misaligned
    assert _call_bwd(p, segs, 1, ch, 2, _grads(2), dout=None) == _lib.RA_ERR_INVALID
    assert _call_bwd(p, segs, 1, ch, 2, _grads(2), dq=None) == _lib.RA_ERR_INVALID
    assert _call_bwd(p, segs, 1, ch, 2, _grads(2), dout=4100) == _lib.RA_ERR_INVALID
    assert _call_bwd(p, segs, 1, ch, 2, _grads(2, ptr=4104)) == _lib.RA_ERR_INVALID
    # the forward's descriptor checks apply
    assert _call_bwd(p, _segs([(200, [(200, 0, 1)])]), 1, ch, 2, _grads(2)) == _lib.RA_ERR_INVALID
    many = [(1, [(1, i, 1)]) for i in range(4097)]
    assert _call_bwd(_problem(Sq=4097), _segs([(4097, [(4097, 0, 1)])]), 1, _chunks(many), 4097,
                     _grads(4097)) == _lib.RA_ERR_UNSUPPORTED


def test_lse_entries_reject_bad_arguments():
    lib = _lib.load()
    assert lib.ra_merge_lse(4, 0, 1, 1, 1, 1, None) == _lib.RA_ERR_INVALID
    assert lib.ra_merge_lse(-1, 8, 1, 1, 1, 1, None) == _lib.RA_ERR_INVALID
    assert lib.ra_merge_lse(4, 8, None, 16, 16, 16, None) == _lib.RA_ERR_INVALID
    assert lib.ra_merge_lse(0, 8, None, None, None, None, None) == _lib.RA_OK
    assert lib.ra_stats_to_lse(4, None, 16, 16, None) == _lib.RA_ERR_INVALID
    assert lib.ra_stats_to_lse(0, None, None, None, None) == _lib.RA_OK


def test_binding_structs_match_the_header_layout(tmp_path):
    """Every ctypes struct of the binding has the size and field offsets the
    C compiler gives the header's struct (a drift would pass garbage through
    the ABI without any error)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    pairs = {"ra_span": _lib.Span, "ra_positions": _lib.Positions, "ra_strides": _lib.Strides,
             "ra_kv_chunk": _lib.KvChunk, "ra_kv_grad": _lib.KvGrad, "ra_q_segment": _lib.QSegment,
             "ra_problem": _lib.Problem}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "ra.h"', "int main(void) {"]
    for cname, cls in pairs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                           str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split("\n")
    got = {tuple(x.split()[:2]): int(x.split()[2]) for x in out if x}
    for cname, cls in pairs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert got[(cname, fname)] == getattr(cls, fname).offset, (cname, fname)
