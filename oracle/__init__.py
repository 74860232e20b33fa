"""CPU oracle of the LatentMoE layer -- TEST INFRASTRUCTURE ONLY.

A ctypes wrapper around lmoe_oracle.c (plain single-threaded C in fp64).
Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package; the CUDA library never calls it and shares no code with
it.  Inputs come from `lmoe_inputs`, which both sides use.

Parity status of each function (how it is pinned to something other than
itself; the tests named live in tests/test_oracle_pins.py):
  e2m1/e4m3/e8m0 decode  -- format closed forms + typed e2m1 grid (golden)
  e2m1/e4m3 encode       -- exhaustive round trips, typed tie cases, brute
                            force nearest-value search in numpy
  scale byte             -- frexp-free integer reference in the test
  quant/dequant MXFP4/8  -- numpy re-implementation from the format spec
  router logits          -- numpy float64 matmul
  top-k + softmax        -- numpy lexsort over all experts; softmax identities
  permute                -- numpy stable argsort + invariants
  MoE tokens (sparse)    -- dense brute force over all experts; numpy
                            float64 SwiGLU on decoded weights; k = E = 1 case
  MoE tokens, FP4 mode   -- numpy float64 SwiGLU with MXFP4 activations
  quant MXFP4 of doubles -- numpy restatement (exact floor(log2) of doubles)
  bf16 rounding          -- torch's fp32 -> bf16 conversion on every kind of
                            fp32 input (no double rounding possible), typed
                            ties / carries / overflow / subnormals (golden),
                            doubles between fp32 neighbours of a midpoint
  linear bf16            -- numpy float64 matmul + bf16 rounding
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lmoe_oracle.c")
_HDR = os.path.join(_HERE, "lmoe_oracle.h")
_LIB_PATH = os.path.join(_HERE, "_lmoe_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Experts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    vp, i32, i64, dbl, u8 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_uint8
    lib.oracle_e2m1_value.argtypes = [u8]
    lib.oracle_e2m1_value.restype = dbl
    lib.oracle_e4m3_value.argtypes = [u8]
    lib.oracle_e4m3_value.restype = dbl
    lib.oracle_e8m0_value.argtypes = [u8]
    lib.oracle_e8m0_value.restype = dbl
    lib.oracle_e2m1_encode.argtypes = [dbl]
    lib.oracle_e2m1_encode.restype = u8
    lib.oracle_e4m3_encode.argtypes = [dbl]
    lib.oracle_e4m3_encode.restype = u8
    lib.oracle_scale_byte.argtypes = [dbl, i32]
    lib.oracle_scale_byte.restype = u8
    lib.oracle_quant_mxfp4.argtypes = [vp, i64, i32, vp, vp]
    lib.oracle_quant_mxfp8.argtypes = [vp, i64, i32, vp, vp]
    lib.oracle_quant_mxfp8_f64.argtypes = [vp, i64, i32, vp, vp]
    lib.oracle_dequant_mxfp4.argtypes = [vp, vp, i64, i32, vp]
    lib.oracle_dequant_mxfp8.argtypes = [vp, vp, i64, i32, vp]
    lib.oracle_router_logits.argtypes = [vp, vp, vp, i32, i32, i32, vp]
    lib.oracle_topk_softmax.argtypes = [vp, i32, i32, i32, vp, vp]
    lib.oracle_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
    lib.oracle_moe_tokens.argtypes = [vp, vp, vp, ctypes.POINTER(_Experts), i32, i32, i32, i32, i32, vp, i32,
                                      vp, vp]
    lib.oracle_expert_ffn_token.argtypes = [vp, ctypes.POINTER(_Experts), i32, i32, i32, vp]
    lib.oracle_moe_dense.argtypes = [vp, vp, vp, ctypes.POINTER(_Experts), i32, i32, i32, i32, i32, vp, i32, vp]
    lib.oracle_linear_bf16.argtypes = [vp, vp, i64, i32, i32, vp]
    lib.oracle_round_bf16.argtypes = [vp, i64, vp]
    lib.oracle_quant_mxfp4_f64.argtypes = [vp, i64, i32, vp, vp]
    lib.oracle_moe_tokens_act.argtypes = [vp, vp, vp, ctypes.POINTER(_Experts), i32, i32, i32, i32, i32, vp, i32,
                                          i32, vp, vp]
    _lib = lib
    return lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- codecs -------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(code)


def e8m0_value(s: int) -> float:
    return _load().oracle_e8m0_value(s)


def e2m1_encode(v: float) -> int:
    return _load().oracle_e2m1_encode(v)


def e4m3_encode(v: float) -> int:
    return _load().oracle_e4m3_encode(v)


def scale_byte(amax: float, emax: int) -> int:
    return _load().oracle_scale_byte(amax, emax)


# ---- block quantisation -------------------------------------------------------

def quant_mxfp4(w: np.ndarray):
    """fp32 [rows, K] -> (codes uint8 [rows, K/2], scales uint8 [rows, K/32])."""
    w = _c(w, np.float32)
    rows, K = w.reshape(-1, w.shape[-1]).shape
    q = np.empty((rows, K // 2), np.uint8)
    s = np.empty((rows, K // 32), np.uint8)
    _load().oracle_quant_mxfp4(_p(w), rows, K, _p(q), _p(s))
    return q.reshape(*w.shape[:-1], K // 2), s.reshape(*w.shape[:-1], K // 32)


def quant_mxfp8(x_bf16: np.ndarray):
    """bf16 bits [rows, K] -> (e4m3 codes [rows, K], scales [rows, K/32])."""
    x = _c(x_bf16, np.uint16)
    rows, K = x.reshape(-1, x.shape[-1]).shape
    q = np.empty((rows, K), np.uint8)
    s = np.empty((rows, K // 32), np.uint8)
    _load().oracle_quant_mxfp8(_p(x), rows, K, _p(q), _p(s))
    return q.reshape(x.shape), s.reshape(*x.shape[:-1], K // 32)


def quant_mxfp8_f64(x: np.ndarray):
    x = _c(x, np.float64)
    rows, K = x.reshape(-1, x.shape[-1]).shape
    q = np.empty((rows, K), np.uint8)
    s = np.empty((rows, K // 32), np.uint8)
    _load().oracle_quant_mxfp8_f64(_p(x), rows, K, _p(q), _p(s))
    return q.reshape(x.shape), s.reshape(*x.shape[:-1], K // 32)


def quant_mxfp4_f64(x: np.ndarray):
    """float64 [rows, K] -> MXFP4 (codes [rows, K/2], scales [rows, K/32])."""
    x = _c(x, np.float64)
    rows, K = x.reshape(-1, x.shape[-1]).shape
    q = np.empty((rows, K // 2), np.uint8)
    s = np.empty((rows, K // 32), np.uint8)
    _load().oracle_quant_mxfp4_f64(_p(x), rows, K, _p(q), _p(s))
    return q.reshape(*x.shape[:-1], K // 2), s.reshape(*x.shape[:-1], K // 32)


def dequant_mxfp4(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.uint8)
    K = q.shape[-1] * 2
    rows = q.size // (K // 2)
    out = np.empty((rows, K), np.float64)
    _load().oracle_dequant_mxfp4(_p(q), _p(s), rows, K, _p(out))
    return out.reshape(*q.shape[:-1], K)


def dequant_mxfp8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.uint8)
    K = q.shape[-1]
    rows = q.size // K
    out = np.empty((rows, K), np.float64)
    _load().oracle_dequant_mxfp8(_p(q), _p(s), rows, K, _p(out))
    return out.reshape(q.shape)


# ---- routing ------------------------------------------------------------------

def router_logits(x_bf16: np.ndarray, Wr: np.ndarray, bias=None) -> np.ndarray:
    x, Wr = _c(x_bf16, np.uint16), _c(Wr, np.float32)
    T, d = x.shape
    E = Wr.shape[0]
    out = np.empty((T, E), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    _load().oracle_router_logits(_p(x), _p(Wr), None if b is None else _p(b), T, d, E, _p(out))
    return out


def topk_softmax(logits: np.ndarray, k: int):
    l = _c(logits, np.float32)
    T, E = l.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _load().oracle_topk_softmax(_p(l), T, E, k, _p(idx), _p(w))
    return idx, w


def permute(idx: np.ndarray, E: int):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    P = T * k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(P, np.int32)
    inv = np.empty(P, np.int32)
    _load().oracle_permute(_p(idx), T, k, E, _p(counts), _p(offsets), _p(perm), _p(inv))
    return counts, offsets, perm, inv


# ---- experts ------------------------------------------------------------------

class Experts:
    """Canonical MXFP4 expert bank (host arrays) as the oracle reads it."""

    def __init__(self, gate_q, gate_s, up_q, up_s, down_q, down_s):
        self.arrays = [_c(a, np.uint8) for a in (gate_q, gate_s, up_q, up_s, down_q, down_s)]
        self.struct = _Experts(*[_p(a) for a in self.arrays])


ACT_MXFP8, ACT_MXFP4 = 1, 2


def moe_tokens(x_bf16, idx, w, experts: Experts, d: int, E: int, I: int, tokens=None, want_f64=False,
               act: int = ACT_MXFP8):
    """The layer on the listed tokens; act = ACT_MXFP8 (x and h rounded to
    MXFP8) or ACT_MXFP4 (the full-FP4 variant: x and h rounded to MXFP4)."""
    x, idx, w = _c(x_bf16, np.uint16), _c(idx, np.int32), _c(w, np.float32)
    T, k = idx.shape
    tok = None if tokens is None else _c(tokens, np.int32)
    ntok = T if tok is None else tok.size
    y = np.empty((ntok, d), np.uint16)
    yf = np.empty((ntok, d), np.float64) if want_f64 else None
    if act == ACT_MXFP8:
        _load().oracle_moe_tokens(_p(x), _p(idx), _p(w), ctypes.byref(experts.struct), T, d, E, k, I,
                                  None if tok is None else _p(tok), ntok, _p(y), None if yf is None else _p(yf))
    else:
        _load().oracle_moe_tokens_act(_p(x), _p(idx), _p(w), ctypes.byref(experts.struct), T, d, E, k, I,
                                      None if tok is None else _p(tok), ntok, act, _p(y),
                                      None if yf is None else _p(yf))
    return (y, yf) if want_f64 else y


def moe_dense(x_bf16, idx, w, experts: Experts, d: int, E: int, I: int, tokens=None):
    x, idx, w = _c(x_bf16, np.uint16), _c(idx, np.int32), _c(w, np.float32)
    T, k = idx.shape
    tok = None if tokens is None else _c(tokens, np.int32)
    ntok = T if tok is None else tok.size
    yf = np.empty((ntok, d), np.float64)
    _load().oracle_moe_dense(_p(x), _p(idx), _p(w), ctypes.byref(experts.struct), T, d, E, k, I,
                             None if tok is None else _p(tok), ntok, _p(yf))
    return yf


def expert_ffn_token(x_row_bf16, experts: Experts, e: int, d: int, I: int) -> np.ndarray:
    x = _c(x_row_bf16, np.uint16)
    out = np.empty(d, np.float64)
    _load().oracle_expert_ffn_token(_p(x), ctypes.byref(experts.struct), e, d, I, _p(out))
    return out


def round_bf16(v) -> np.ndarray:
    """bf16 bits of float64 values, rounded once to nearest even."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_round_bf16(_p(v), v.size, _p(out))
    return out


def linear_bf16(x_bf16: np.ndarray, W_bf16: np.ndarray) -> np.ndarray:
    x, W = _c(x_bf16, np.uint16), _c(W_bf16, np.uint16)
    rows, K = x.shape
    N = W.shape[0]
    out = np.empty((rows, N), np.uint16)
    _load().oracle_linear_bf16(_p(x), _p(W), rows, K, N, _p(out))
    return out


# ---- whole layer --------------------------------------------------------------

def quantize_experts(wl, e0: int = 0, e1: int | None = None, experts=None):
    """Oracle-side MXFP4 quantisation of the generator's fp32 expert weights.

    Returns canonical arrays for all E experts; only [e0, e1) (or the listed
    `experts`) are filled, the rest stay zero (never read when not routed to)."""
    import lmoe_inputs as gen
    E, I, d = wl.E, wl.I, wl.d
    gq = np.zeros((E, I, d // 2), np.uint8); gs = np.zeros((E, I, d // 32), np.uint8)
    uq = np.zeros((E, I, d // 2), np.uint8); us = np.zeros((E, I, d // 32), np.uint8)
    dq = np.zeros((E, d, I // 2), np.uint8); ds = np.zeros((E, d, I // 32), np.uint8)
    ids = list(range(e0, E if e1 is None else e1)) if experts is None else sorted(set(int(e) for e in experts))
    for e in ids:
        gq[e], gs[e] = quant_mxfp4(gen.expert_f32(wl, "gate", e, e + 1)[0])
        uq[e], us[e] = quant_mxfp4(gen.expert_f32(wl, "up", e, e + 1)[0])
        dq[e], ds[e] = quant_mxfp4(gen.expert_f32(wl, "down", e, e + 1)[0])
    return Experts(gq, gs, uq, us, dq, ds)
