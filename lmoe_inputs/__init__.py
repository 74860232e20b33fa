"""Seeded synthetic inputs for the LatentMoE layer.

This package only *generates* input tensors (numpy arrays on the host); it
contains none of the layer's arithmetic.  The CUDA library and the CPU oracle
are both fed from it, so they see byte-identical inputs.

Workloads (shapes follow the pages' model: 896 experts, top-16, a 3584-wide
latent space, MXFP4 expert weights; the intermediate width is not stated on
the pages and is fixed per workload here):

  tiny     T=8,     d=512,  I=64   correctness-sized layer
  decode   T=64,    d=3584, I=512  decode-shaped batch, weight-bandwidth bound
  prefill  T=8192,  d=3584, I=512  prefill chunk, about 146 tokens per expert
  skewed   as prefill, router logits biased by beta*ln(Zipf(1.2) popularity)
  block    T=32768, hidden 7168 -> latent 3584 -> experts -> hidden 7168

Value distributions: activations ~ N(0, 1) rounded to bf16; router weights
fp32 ~ N(0, 1/sqrt(d)); expert and projection weights fp32 ~ N(0,
1/sqrt(fan_in)) (fan_in = d for gate/up, I for down, hidden or d for the
projections; sigma is the standard deviation).  Every tensor has its own
stream of the counter-based generator in gen.c, so any expert's weights can
be produced on their own.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_lmoe_gen.so")
_lib = None

# one stream per tensor
STREAM_X = 1
STREAM_WR = 2
STREAM_WG = 3
STREAM_WU = 4
STREAM_WD = 5
STREAM_XH = 6
STREAM_WIN = 7
STREAM_WOUT = 8


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library next to it (gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lpthread", "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, dbl, i32 = ctypes.c_uint64, ctypes.c_double, ctypes.c_int
        vp = ctypes.c_void_p
        lib.lmoe_gen_normal_f32.argtypes = [u64, u64, u64, u64, dbl, vp, i32]
        lib.lmoe_gen_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, vp, i32]
        lib.lmoe_gen_raw_u64.argtypes = [u64, u64, u64, u64, vp]
        lib.lmoe_gen_det_log.argtypes = [dbl]
        lib.lmoe_gen_det_log.restype = dbl
        lib.lmoe_gen_det_exp.argtypes = [dbl]
        lib.lmoe_gen_det_exp.restype = dbl
        lib.lmoe_gen_det_sincos_turn.argtypes = [dbl, vp, vp]
        lib.lmoe_gen_zipf_bias.argtypes = [i32, dbl, dbl, vp]
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_f32(seed: int, stream: int, start: int, n: int, sigma: float, out=None) -> np.ndarray:
    out = np.empty(n, np.float32) if out is None else out
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    _load().lmoe_gen_normal_f32(seed, stream, start, n, sigma, out.ctypes.data, _threads())
    return out


def normal_bf16(seed: int, stream: int, start: int, n: int, sigma: float, out=None) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, sigma) samples rounded to nearest even."""
    out = np.empty(n, np.uint16) if out is None else out
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    _load().lmoe_gen_normal_bf16(seed, stream, start, n, sigma, out.ctypes.data, _threads())
    return out


def raw_u64(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().lmoe_gen_raw_u64(seed, stream, start, n, out.ctypes.data)
    return out


def det_log(x: float) -> float:
    return _load().lmoe_gen_det_log(x)


def det_exp(x: float) -> float:
    return _load().lmoe_gen_det_exp(x)


def det_sincos_turn(u: float):
    s, c = ctypes.c_double(), ctypes.c_double()
    _load().lmoe_gen_det_sincos_turn(u, ctypes.byref(s), ctypes.byref(c))
    return s.value, c.value


def zipf_bias(E: int, s: float, beta: float) -> np.ndarray:
    out = np.empty(E, np.float32)
    _load().lmoe_gen_zipf_bias(E, s, beta, out.ctypes.data)
    return out


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    I: int
    E: int = 896
    k: int = 16
    seed: int = 0
    hidden: int = 0          # > 0: hidden-width block with bf16 projections around the layer
    zipf_s: float = 0.0      # > 0: skewed routing bias beta*ln p_zipf(e)
    zipf_beta: float = 0.0
    note: str = field(default="", compare=False)

    @property
    def P(self) -> int:
        return self.T * self.k


WORKLOADS = {
    "tiny": Workload("tiny", T=8, d=512, I=64, note="T=8, d=512, I=64"),
    "decode": Workload("decode", T=64, d=3584, I=512, note="T=64 decode-shaped batch"),
    "decode1": Workload("decode1", T=1, d=3584, I=512, note="T=1 batch-1 decode step (16 experts)"),
    "decode16": Workload("decode16", T=16, d=3584, I=512, note="T=16 small-batch decode step"),
    "prefill": Workload("prefill", T=8192, d=3584, I=512, note="T=8192 prefill chunk"),
    "skewed": Workload("skewed", T=8192, d=3584, I=512, zipf_s=1.2, zipf_beta=0.18,
                       note="T=8192, Zipf(1.2) popularity bias, beta=0.18"),
    "block": Workload("block", T=32768, d=3584, I=512, hidden=7168,
                      note="T=32768, hidden 7168 -> latent 3584 -> experts -> 7168"),
}


def custom(name: str, T: int, d: int, I: int, E: int = 896, k: int = 16, seed: int = 0, **kw) -> Workload:
    return Workload(name, T=T, d=d, I=I, E=E, k=k, seed=seed, **kw)


# ---- tensors of a workload ----------------------------------------------------

def x_bf16(w: Workload, t0: int = 0, t1: int | None = None) -> np.ndarray:
    """Latent activations [T, d] as bf16 bits, N(0, 1)."""
    t1 = w.T if t1 is None else t1
    return normal_bf16(w.seed, STREAM_X, t0 * w.d, (t1 - t0) * w.d, 1.0).reshape(t1 - t0, w.d)


def router_f32(w: Workload) -> np.ndarray:
    """Router weights W_r [E, d], fp32, N(0, 1/sqrt(d))."""
    return normal_f32(w.seed, STREAM_WR, 0, w.E * w.d, 1.0 / math.sqrt(w.d)).reshape(w.E, w.d)


def router_bias(w: Workload):
    """Per-expert logit bias (skewed workload) or None."""
    if w.zipf_s <= 0.0:
        return None
    return zipf_bias(w.E, w.zipf_s, w.zipf_beta)


def expert_f32(w: Workload, which: str, e0: int, e1: int) -> np.ndarray:
    """fp32 weights of experts [e0, e1): gate/up [n, I, d] (sigma 1/sqrt(d)),
    down [n, d, I] (sigma 1/sqrt(I))."""
    if which in ("gate", "up"):
        rows, K, stream = w.I, w.d, STREAM_WG if which == "gate" else STREAM_WU
    elif which == "down":
        rows, K, stream = w.d, w.I, STREAM_WD
    else:
        raise ValueError(which)
    per = rows * K
    a = normal_f32(w.seed, stream, e0 * per, (e1 - e0) * per, 1.0 / math.sqrt(K))
    return a.reshape(e1 - e0, rows, K)


def hidden_bf16(w: Workload, t0: int = 0, t1: int | None = None) -> np.ndarray:
    """Block input [T, hidden] as bf16 bits, N(0, 1)."""
    t1 = w.T if t1 is None else t1
    return normal_bf16(w.seed, STREAM_XH, t0 * w.hidden, (t1 - t0) * w.hidden, 1.0).reshape(t1 - t0, w.hidden)


def proj_in_bf16(w: Workload) -> np.ndarray:
    """Down-projection W_in [d, hidden] as bf16 bits, N(0, 1/sqrt(hidden))."""
    return normal_bf16(w.seed, STREAM_WIN, 0, w.d * w.hidden, 1.0 / math.sqrt(w.hidden)).reshape(w.d, w.hidden)


def proj_out_bf16(w: Workload) -> np.ndarray:
    """Up-projection W_out [hidden, d] as bf16 bits, N(0, 1/sqrt(d))."""
    return normal_bf16(w.seed, STREAM_WOUT, 0, w.hidden * w.d, 1.0 / math.sqrt(w.d)).reshape(w.hidden, w.d)
