"""The C-ABI library: it builds, loads, exports every entry point the public
header declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lmoe.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lmoe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from top_routing_mxfp4_gb300 import build
    return ctypes.CDLL(build.build())


def test_header_declares_the_layer_calls():
    names = _declared()
    for n in ("lmoe_quant_mxfp4", "lmoe_route", "lmoe_permute", "lmoe_expert_ffn", "lmoe_combine", "lmoe_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_side_argument_checks(lib):
    from top_routing_mxfp4_gb300 import lmoe
    D = lmoe.Dims
    ws_size = lib.lmoe_workspace_size
    ws_size.restype = ctypes.c_size_t
    ws_size.argtypes = [ctypes.POINTER(D)]
    assert ws_size(ctypes.byref(D(64, 3584, 896, 16, 512, 1))) > 0
    for bad in (D(8, 500, 896, 16, 64, 1), D(8, 512, 896, 33, 64, 1), D(8, 512, 8, 16, 64, 1),
                D(-1, 512, 896, 16, 64, 1), D(8, 512, 896, 16, 48, 1), D(8, 512, 4096, 16, 64, 1)):
        assert ws_size(ctypes.byref(bad)) == 0
    fwd = lib.lmoe_forward
    fwd.restype = ctypes.c_int
    vp = ctypes.c_void_p
    fwd.argtypes = [vp, vp, vp, ctypes.POINTER(lmoe.ExpertWeights), ctypes.POINTER(D), vp, vp, vp, vp, vp,
                    ctypes.c_size_t, vp]
    good = D(8, 512, 896, 16, 64, 1)
    # null weights / null pointers / bad dims are refused before any launch
    assert fwd(None, None, None, None, ctypes.byref(good), None, None, None, None, None, 0, None) == lmoe.ERR_INVALID_ARG
    assert fwd(None, None, None, None, ctypes.byref(D(8, 500, 896, 16, 64, 1)), None, None, None, None, None, 0,
               None) == lmoe.ERR_INVALID_ARG
    # unsupported activation format
    assert fwd(None, None, None, None, ctypes.byref(D(8, 512, 896, 16, 64, 0)), None, None, None, None, None, 0,
               None) == lmoe.ERR_UNSUPPORTED
    # weights in the canonical layout are refused by the expert GEMMs
    W = lmoe.ExpertWeights(256, 256, 256, 256, 256, 256, lmoe.LAYOUT_CANONICAL)
    assert fwd(ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.byref(W), ctypes.byref(good),
               ctypes.c_void_p(256), None, None, None, ctypes.c_void_p(256), 1 << 30, None) == lmoe.ERR_INVALID_ARG
    # too small a workspace
    W = lmoe.ExpertWeights(256, 256, 256, 256, 256, 256, lmoe.LAYOUT_TC)
    assert fwd(ctypes.c_void_p(256), ctypes.c_void_p(256), None, ctypes.byref(W), ctypes.byref(good),
               ctypes.c_void_p(256), None, None, None, ctypes.c_void_p(256), 16, None) == lmoe.ERR_WORKSPACE
    # empty batch is a no-op
    assert fwd(None, None, None, None, ctypes.byref(D(0, 512, 896, 16, 64, 1)), None, None, None, None, None, 0,
               None) == lmoe.OK


def test_expert_ffn_argument_checks(lib):
    """The stage entry point refuses null or misaligned operands and a short
    workspace before any launch."""
    from top_routing_mxfp4_gb300 import lmoe
    D = lmoe.Dims
    good = D(64, 3584, 896, 16, 512, 1)
    size = lib.lmoe_expert_ffn_workspace_size
    size.restype = ctypes.c_size_t
    size.argtypes = [ctypes.POINTER(D)]
    need = size(ctypes.byref(good))
    assert need > 0
    # a larger batch never needs less scratch
    assert size(ctypes.byref(D(8192, 3584, 896, 16, 512, 1))) > need
    ffn = lib.lmoe_expert_ffn
    ffn.restype = ctypes.c_int
    vp = ctypes.c_void_p
    ffn.argtypes = [vp, vp, ctypes.POINTER(lmoe.ExpertWeights), vp, vp, vp, ctypes.POINTER(D), vp, vp,
                    ctypes.c_size_t, vp]
    W = lmoe.ExpertWeights(256, 256, 256, 256, 256, 256, lmoe.LAYOUT_TC)
    p = ctypes.c_void_p(4096)

    def call(xq=p, xs=p, ws=p, ws_bytes=need, dims=good):
        return ffn(xq, xs, ctypes.byref(W), p, p, p, ctypes.byref(dims), p, ws, ws_bytes, None)

    assert call(xq=None) == lmoe.ERR_INVALID_ARG
    assert call(xs=None) == lmoe.ERR_INVALID_ARG
    assert call(xq=ctypes.c_void_p(4104)) == lmoe.ERR_INVALID_ARG   # codes not 16-byte aligned
    assert call(xs=ctypes.c_void_p(4100)) == lmoe.ERR_INVALID_ARG   # scales not 16-byte aligned
    assert call(ws_bytes=need - 1) == lmoe.ERR_WORKSPACE
    assert call(ws=ctypes.c_void_p(4096 + 16)) == lmoe.ERR_WORKSPACE  # workspace not 256-byte aligned
    assert call(dims=D(0, 3584, 896, 16, 512, 1)) == lmoe.OK          # empty batch: nothing to do


def test_mxfp4_byte_counts(lib):
    from top_routing_mxfp4_gb300 import lmoe
    assert lmoe.mxfp4_bytes(896, 512, 3584, lmoe.LAYOUT_CANONICAL) == (896 * 512 * 1792, 896 * 512 * 112)
    assert lmoe.mxfp4_bytes(896, 512, 3584, lmoe.LAYOUT_TC) == (896 * 512 * 1792, 896 * 512 * 112)
    # K padded to 128, rows to whole 128-row atoms
    assert lmoe.mxfp4_bytes(2, 64, 64, lmoe.LAYOUT_TC) == (2 * 64 * 64, 2 * 1 * 1 * 512)
    with pytest.raises(ValueError):
        lmoe.mxfp4_bytes(1, 8, 48, lmoe.LAYOUT_TC)


@pytest.mark.parametrize("T,tile", [(1, 16), (64, 16), (512, 32), (2048, 96)])
def test_forward_workspace_views_layout(lib, T, tile):
    """lmoe_forward_workspace_views is host arithmetic: at every token-tile
    shape the views lie inside lmoe_workspace_size and do not overlap; the
    split-K arrival counters (int32 [128][4], zeroed 16 bytes at a time by the
    schedule) exist at 16-token tiles only and are 16-byte aligned."""
    from top_routing_mxfp4_gb300 import lmoe
    d, E, k, I = 3584, 896, 16, 512
    ws_size = lib.lmoe_workspace_size
    ws_size.restype = ctypes.c_size_t
    ws_size.argtypes = [ctypes.POINTER(lmoe.Dims)]
    old = lmoe.small_batch_pairs()
    lmoe.set_small_batch_pairs(0)  # the tensor-core path's layout
    try:
        total = ws_size(ctypes.byref(lmoe.Dims(T, d, E, k, I, 1)))
        v = lmoe.forward_workspace_views(T, d, E, k, I)
    finally:
        lmoe.set_small_batch_pairs(old)
    assert v.path == 0 and v.tile_tokens == tile
    P = T * k
    regions = {"xq": (v.xq, v.rows * d), "hq": (v.hq, v.rows * I), "dst_row": (v.dst_row, 4 * P),
               "code_row": (v.code_row, 4 * P)}
    if tile == 16:
        assert v.ksplit >= 0 and v.ksplit % 16 == 0
        regions["ksplit"] = (v.ksplit, 128 * 4 * 4)
    else:
        assert v.ksplit == -1
    spans = sorted(regions.items(), key=lambda kv: kv[1][0])
    for name, (off, size) in spans:
        assert 0 <= off and off + size <= total, name
    for (n0, (o0, s0)), (n1, (o1, _)) in zip(spans, spans[1:]):
        assert o0 + s0 <= o1, f"{n0} overlaps {n1}"
