"""ctypes binding of liblmoe.so, the LatentMoE layer's C ABI (include/lmoe.h).

Argument marshalling only: every function takes torch CUDA tensors, checks
shapes and dtypes, and passes `data_ptr()` plus the current CUDA stream to
the C entry point of the same name.  All arithmetic runs in the library's
CUDA kernels.  Importing this module fails loudly when the library has not
been built (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# LMOE_LIBRARY selects another build of the same library (e.g. a trace build)
LIB_PATH = os.environ.get("LMOE_LIBRARY") or os.path.join(_PKG, "liblmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
                      "or `python top_routing_mxfp4_gb300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_DEVICE_CHECK = -5
ERR_TIMEOUT = -6
ACT_MXFP8 = 1
ACT_MXFP4 = 2
LAYOUT_CANONICAL = 0
LAYOUT_TC = 1


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("I", ctypes.c_int32), ("act", ctypes.c_int32)]


class ExpertWeights(ctypes.Structure):
    _fields_ = [("gate_q", ctypes.c_void_p), ("gate_s", ctypes.c_void_p), ("up_q", ctypes.c_void_p),
                ("up_s", ctypes.c_void_p), ("down_q", ctypes.c_void_p), ("down_s", ctypes.c_void_p),
                ("layout", ctypes.c_int32)]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_DP, _WP = ctypes.POINTER(Dims), ctypes.POINTER(ExpertWeights)


def _sig(name, restype, *argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_lib_version = _sig("lmoe_version", ctypes.c_char_p)
_status_string = _sig("lmoe_status_string", ctypes.c_char_p, ctypes.c_int)
_mxfp4_bytes = _sig("lmoe_mxfp4_bytes", _sz, _i64, _i32, _i32, _i32, ctypes.POINTER(_sz))
_quant_mxfp4 = _sig("lmoe_quant_mxfp4", ctypes.c_int, _vp, _i64, _i32, _i32, _vp, _vp, _i32, _vp)
_quant_mxfp8 = _sig("lmoe_quant_mxfp8", ctypes.c_int, _vp, _i64, _i32, _vp, _vp, _vp)
_repack_mxfp4 = _sig("lmoe_repack_mxfp4", ctypes.c_int, _vp, _vp, _i64, _i32, _i32, _vp, _vp, _vp)
_scale_hist = _sig("lmoe_mxfp4_scale_histogram", ctypes.c_int, _vp, _i64, _i32, _i32, _i32, _vp, _vp)
_route = _sig("lmoe_route", ctypes.c_int, _vp, _vp, _vp, _DP, _vp, _vp, _vp, _vp, _sz, _vp)
_router_bytes = _sig("lmoe_router_prepared_bytes", _sz, _i32, _i32)
_prepare_router = _sig("lmoe_prepare_router", ctypes.c_int, _vp, _i32, _i32, _vp, _vp)
_route_ws = _sig("lmoe_route_workspace_size", _sz, _DP)
_topk = _sig("lmoe_topk_from_logits", ctypes.c_int, _vp, _DP, _vp, _vp, _vp)
_perm_ws = _sig("lmoe_permute_workspace_size", _sz, _DP)
_permute = _sig("lmoe_permute", ctypes.c_int, _vp, _DP, _vp, _vp, _vp, _vp, _vp, _sz, _vp)
_permute_noalloc = _sig("lmoe_permute_noalloc", ctypes.c_int, _vp, _DP, _vp, _vp, _vp, _vp, _vp, _vp)
PERMUTE_NOALLOC_MAX_PAIRS = 524288
_ffn_ws = _sig("lmoe_expert_ffn_workspace_size", _sz, _DP)
_ffn = _sig("lmoe_expert_ffn", ctypes.c_int, _vp, _vp, _WP, _vp, _vp, _vp, _DP, _vp, _vp, _sz, _vp)
_combine = _sig("lmoe_combine", ctypes.c_int, _vp, _vp, _DP, _vp, _vp)
_ws_size = _sig("lmoe_workspace_size", _sz, _DP)
_forward = _sig("lmoe_forward", ctypes.c_int, _vp, _vp, _vp, _WP, _DP, _vp, _vp, _vp, _vp, _vp, _sz, _vp)
_linear = _sig("lmoe_linear_bf16", ctypes.c_int, _vp, _vp, _i64, _i32, _i32, _vp, _vp)
_block_ws = _sig("lmoe_block_workspace_size", _sz, _DP, _i32)
_forward_block = _sig("lmoe_forward_block", ctypes.c_int, _vp, _vp, _vp, _vp, _WP, _vp, _DP, _i32, _vp, _vp, _vp, _vp,
                      _vp, _vp, _vp, _sz, _vp)
_last_status = _sig("lmoe_last_device_status", ctypes.c_int, _vp, ctypes.POINTER(_i32))
_clear_status = _sig("lmoe_clear_device_status", ctypes.c_int, _vp, _vp)
_set_events = _sig("lmoe_set_stage_events", ctypes.c_int, ctypes.POINTER(_vp), _i32)
_kernel_count = _sig("lmoe_forward_kernel_count", _i32, _DP)


class FfnViews(ctypes.Structure):
    _fields_ = [("xq", _i64), ("xs", _i64), ("hq", _i64), ("hs", _i64), ("dst_row", _i64), ("rows", _i64),
                ("tile_tokens", _i32), ("slot_rows", _i32), ("path", _i32), ("code_row", _i64), ("ksplit", _i64)]


_ws_views = _sig("lmoe_forward_workspace_views", ctypes.c_int, _DP, ctypes.POINTER(FfnViews))
_set_hcap = _sig("lmoe_set_h_capture", ctypes.c_int, _vp, _sz)
_set_wait_test = _sig("lmoe_set_wait_test", ctypes.c_int, _i32, _i64)
_set_small = _sig("lmoe_set_small_batch_pairs", ctypes.c_int, _i32)


def set_wait_test(stall_first_fill: bool, wait_limit_cycles: int = 0):
    """Failure-path test hook of the expert GEMMs' bounded waits
    (lmoe_set_wait_test); (False, 0) restores the normal behaviour."""
    _check(_set_wait_test(1 if stall_first_fill else 0, int(wait_limit_cycles)), "lmoe_set_wait_test")
_get_small = _sig("lmoe_small_batch_pairs", _i32)
SMALL_BATCH_PAIRS_DEFAULT = 0


def set_small_batch_pairs(max_pairs: int):
    """Batches of at most this many pairs (T * k, at most 8 tokens) run the
    small-batch path of lmoe_forward; 0 sends every batch to the tensor-core
    path.  Process-wide."""
    _check(_set_small(int(max_pairs)), "lmoe_set_small_batch_pairs")


def small_batch_pairs() -> int:
    return int(_get_small())


def forward_workspace_views(T: int, d: int, E: int, k: int, I: int) -> FfnViews:
    """Byte offsets of the expert GEMMs' MXFP8 operands inside lmoe_forward's
    workspace (diagnostics)."""
    v = FfnViews()
    D = dims(T, d, E, k, I)
    _check(_ws_views(ctypes.byref(D), ctypes.byref(v)), "lmoe_forward_workspace_views")
    return v


def set_h_capture(buf):
    """Diagnostics: a float32 CUDA tensor that later forward calls fill with
    the fp32 h values their gate/up GEMM rounds to MXFP8; None clears it."""
    if buf is None:
        _check(_set_hcap(None, 0), "lmoe_set_h_capture")
        return
    if buf.dtype != torch.float32 or not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("h capture buffer: contiguous CUDA float32 tensor expected")
    _check(_set_hcap(_ptr(buf), buf.numel() * 4), "lmoe_set_h_capture")


def forward_kernel_count(T: int, d: int, E: int, k: int, I: int) -> int:
    D = dims(T, d, E, k, I)
    return int(_kernel_count(ctypes.byref(D)))
NUM_STAGE_EVENTS = 7
STAGES = ("route", "permute", "act_quant", "gate_up", "down", "combine")


def set_stage_events(events):
    """Record these torch.cuda.Event objects at lmoe_forward's stage boundaries
    (start, after route, permute, activation scatter, gate/up GEMM, down GEMM,
    combine); None clears the hook."""
    if events is None:
        _check(_set_events(None, 0), "lmoe_set_stage_events")
        return
    assert len(events) == NUM_STAGE_EVENTS
    arr = (_vp * NUM_STAGE_EVENTS)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(_set_events(arr, NUM_STAGE_EVENTS), "lmoe_set_stage_events")


class LmoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def status_string(code: int) -> str:
    return _status_string(code).decode()


def version() -> str:
    return _lib_version().decode()


def _check(code: int, what: str):
    if code != OK:
        raise LmoeError(code, what)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous CUDA {dtype} {tuple(shape)}, got {t.dtype} "
                         f"{tuple(t.shape)} on {t.device}")


def dims(T: int, d: int, E: int, k: int, I: int, act: int = ACT_MXFP8) -> Dims:
    return Dims(T, d, E, k, I, act)


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---- load-time conversion ----------------------------------------------------------

def mxfp4_bytes(nmat: int, rows: int, K: int, layout: int):
    sb = _sz()
    qb = _mxfp4_bytes(nmat, rows, K, layout, ctypes.byref(sb))
    if qb == 0 and nmat > 0:
        raise ValueError("bad MXFP4 matrix sizes")
    return int(qb), int(sb.value)


def quant_mxfp4(w: torch.Tensor, layout: int = LAYOUT_TC, q=None, s=None, stream=None):
    """fp32 [nmat, rows, K] (or [rows, K]) -> (codes, scales) as flat uint8 tensors."""
    w3 = w if w.dim() == 3 else w.unsqueeze(0)
    nmat, rows, K = w3.shape
    _need(w3, torch.float32, (nmat, rows, K), "w")
    qb, sb = mxfp4_bytes(nmat, rows, K, layout)
    q = _empty(qb, torch.uint8, w.device) if q is None else q
    s = _empty(sb, torch.uint8, w.device) if s is None else s
    assert q.numel() >= qb and s.numel() >= sb
    _check(_quant_mxfp4(_ptr(w3), nmat, rows, K, _ptr(q), _ptr(s), layout, _stream(stream)), "lmoe_quant_mxfp4")
    return q, s


def repack_mxfp4(q: torch.Tensor, s: torch.Tensor, nmat: int, rows: int, K: int, q_tc=None, s_tc=None, stream=None):
    """Canonical MXFP4 bytes (uint8 codes [nmat*rows*K/2], scales
    [nmat*rows*K/32], flat or shaped) -> the tensor-core layout, as flat uint8
    tensors (byte rearrangement; lmoe_repack_mxfp4)."""
    qb, sb = mxfp4_bytes(nmat, rows, K, LAYOUT_TC)
    _need(q, torch.uint8, q.shape, "q")
    _need(s, torch.uint8, s.shape, "s")
    if q.numel() != nmat * rows * K // 2 or s.numel() != nmat * rows * K // 32:
        raise ValueError("canonical MXFP4 arrays of the wrong size")
    q_tc = _empty(qb, torch.uint8, q.device) if q_tc is None else q_tc
    s_tc = _empty(sb, torch.uint8, q.device) if s_tc is None else s_tc
    if q_tc.numel() < qb or s_tc.numel() < sb:
        raise ValueError("tensor-core layout destination too small")
    _check(_repack_mxfp4(_ptr(q), _ptr(s), nmat, rows, K, _ptr(q_tc), _ptr(s_tc), _stream(stream)),
           "lmoe_repack_mxfp4")
    return q_tc, s_tc


def scale_histogram(s: torch.Tensor, nmat: int, rows: int, K: int, layout: int = LAYOUT_TC, stream=None):
    """Per-matrix counts of each E8M0 scale byte: int32-viewed uint32 [nmat, 256]."""
    _need(s, torch.uint8, s.shape, "s")
    hist = _empty((nmat, 256), torch.int32, s.device)
    _check(_scale_hist(_ptr(s), nmat, rows, K, layout, _ptr(hist), _stream(stream)), "lmoe_mxfp4_scale_histogram")
    return hist


def quant_mxfp8(x: torch.Tensor, stream=None):
    """bf16 [rows, K] -> (e4m3 codes uint8 [rows, K], scales uint8 [rows, K/32])."""
    rows, K = x.shape
    _need(x, torch.bfloat16, (rows, K), "x")
    q = _empty((rows, K), torch.uint8, x.device)
    s = _empty((rows, K // 32), torch.uint8, x.device)
    _check(_quant_mxfp8(_ptr(x), rows, K, _ptr(q), _ptr(s), _stream(stream)), "lmoe_quant_mxfp8")
    return q, s


class ExpertBank:
    """An expert bank in the tensor-core MXFP4 layout, resident on the device.

    Built matrix by matrix from fp32 weights (load-time conversion), so the
    fp32 copy of the whole bank never has to exist on the device."""

    def __init__(self, E: int, d: int, I: int, device):
        self.E, self.d, self.I = E, d, I
        self.device = torch.device(device)
        gqb, gsb = mxfp4_bytes(E, I, d, LAYOUT_TC)
        dqb, dsb = mxfp4_bytes(E, d, I, LAYOUT_TC)
        self.gate_q, self.gate_s = _empty(gqb, torch.uint8, device), _empty(gsb, torch.uint8, device)
        self.up_q, self.up_s = _empty(gqb, torch.uint8, device), _empty(gsb, torch.uint8, device)
        self.down_q, self.down_s = _empty(dqb, torch.uint8, device), _empty(dsb, torch.uint8, device)
        self._struct = None

    @property
    def nbytes(self) -> int:
        return sum(t.numel() for t in (self.gate_q, self.gate_s, self.up_q, self.up_s, self.down_q, self.down_s))

    def load(self, which: str, e0: int, w: torch.Tensor, stream=None):
        """Quantise fp32 weights of experts [e0, e0 + w.shape[0]) into the bank."""
        n = w.shape[0]
        if which in ("gate", "up"):
            rows, K = self.I, self.d
        else:
            rows, K = self.d, self.I
        qb1, sb1 = mxfp4_bytes(1, rows, K, LAYOUT_TC)
        q = getattr(self, which + "_q")[e0 * qb1:(e0 + n) * qb1]
        s = getattr(self, which + "_s")[e0 * sb1:(e0 + n) * sb1]
        quant_mxfp4(w.reshape(n, rows, K), LAYOUT_TC, q, s, stream)

    def load_mxfp4(self, which: str, e0: int, q: torch.Tensor, s: torch.Tensor, stream=None):
        """Copy a checkpoint's canonical MXFP4 matrices of experts [e0, e0 + n)
        into the bank (lmoe_repack_mxfp4).  q, s: uint8 codes [n, rows, K/2]
        and scales [n, rows, K/32] on the device, e.g. a staging buffer the
        caller refills chunk by chunk."""
        rows, K = (self.I, self.d) if which in ("gate", "up") else (self.d, self.I)
        n = q.shape[0]
        qb1, sb1 = mxfp4_bytes(1, rows, K, LAYOUT_TC)
        qd = getattr(self, which + "_q")[e0 * qb1:(e0 + n) * qb1]
        sd = getattr(self, which + "_s")[e0 * sb1:(e0 + n) * sb1]
        repack_mxfp4(q, s, n, rows, K, qd, sd, stream)

    def scale_histograms(self, stream=None):
        """E8M0 scale-byte counts per expert matrix: {gate, up, down}: [E, 256]."""
        return {w: scale_histogram(getattr(self, w + "_s"), self.E, *((self.I, self.d) if w != "down" else
                                                                       (self.d, self.I)), LAYOUT_TC, stream)
                for w in ("gate", "up", "down")}

    def struct(self) -> ExpertWeights:
        if self._struct is None:
            self._struct = ExpertWeights(self.gate_q.data_ptr(), self.gate_s.data_ptr(), self.up_q.data_ptr(),
                                         self.up_s.data_ptr(), self.down_q.data_ptr(), self.down_s.data_ptr(),
                                         LAYOUT_TC)
        return self._struct


# ---- stages ------------------------------------------------------------------------

def prepare_router(Wr, stream=None):
    """fp32 router weights [E, d] -> the three bf16 planes [3, E, d] the router
    GEMM reads (their sum is Wr exactly)."""
    E, d = Wr.shape
    _need(Wr, torch.float32, (E, d), "Wr")
    if int(_router_bytes(E, d)) == 0:
        raise ValueError(f"router weights [{E}, {d}]: d must be a multiple of 64")
    Wr3 = _empty((3, E, d), torch.bfloat16, Wr.device)
    _check(_prepare_router(_ptr(Wr), E, d, _ptr(Wr3), _stream(stream)), "lmoe_prepare_router")
    return Wr3


def route(x, Wr, k: int, bias=None, stream=None, Wr3=None):
    """Router + top-k + softmax.  Wr: fp32 [E, d] (prepared on the fly) or
    Wr3: prepared planes [3, E, d]."""
    T, d = x.shape
    if Wr3 is None:
        Wr3 = prepare_router(Wr, stream)
    E = Wr3.shape[1]
    _need(x, torch.bfloat16, (T, d), "x")
    _need(Wr3, torch.bfloat16, (3, E, d), "Wr3")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    D = dims(T, d, E, k, 32)
    logits = _empty((T, E), torch.float32, x.device)
    idx = _empty((T, k), torch.int32, x.device)
    w = _empty((T, k), torch.float32, x.device)
    ws = workspace(_route_ws(ctypes.byref(D)), x.device)
    _check(_route(_ptr(x), _ptr(Wr3), _ptr(bias), ctypes.byref(D), _ptr(logits), _ptr(idx), _ptr(w), _ptr(ws),
                  ws.numel(), _stream(stream)), "lmoe_route")
    return logits, idx, w


def topk_from_logits(logits, k: int, stream=None):
    T, E = logits.shape
    _need(logits, torch.float32, (T, E), "logits")
    D = dims(T, 128, E, k, 32)
    idx = _empty((T, k), torch.int32, logits.device)
    w = _empty((T, k), torch.float32, logits.device)
    _check(_topk(_ptr(logits), ctypes.byref(D), _ptr(idx), _ptr(w), _stream(stream)), "lmoe_topk_from_logits")
    return idx, w


def permute_workspace_size(T: int, E: int, k: int) -> int:
    D = dims(T, 128, E, k, 32)
    return int(_perm_ws(ctypes.byref(D)))


def permute(idx, E: int, ws=None, stream=None):
    T, k = idx.shape
    _need(idx, torch.int32, (T, k), "topk_idx")
    D = dims(T, 128, E, k, 32)
    dev = idx.device
    counts = _empty(E, torch.int32, dev)
    offsets = _empty(E + 1, torch.int32, dev)
    perm = _empty(T * k, torch.int32, dev)
    inv = _empty(T * k, torch.int32, dev)
    ws = workspace(_perm_ws(ctypes.byref(D)), dev) if ws is None else ws
    _check(_permute(_ptr(idx), ctypes.byref(D), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(ws),
                    ws.numel(), _stream(stream)), "lmoe_permute")
    return counts, offsets, perm, inv, ws


def permute_noalloc(idx, E: int, out=None, stream=None):
    """lmoe_permute_noalloc: the permute with no workspace (the library's fixed
    device array holds the scratch).  `out` may pass preallocated
    (counts, offsets, perm, inv, device_status) tensors, so the call itself
    allocates nothing."""
    T, k = idx.shape
    _need(idx, torch.int32, (T, k), "topk_idx")
    D = dims(T, 128, E, k, 32)
    dev = idx.device
    if out is None:
        out = (_empty(E, torch.int32, dev), _empty(E + 1, torch.int32, dev), _empty(T * k, torch.int32, dev),
               _empty(T * k, torch.int32, dev), _empty(1, torch.int32, dev))
    counts, offsets, perm, inv, status = out
    for t, shape, name in ((counts, (E,), "counts"), (offsets, (E + 1,), "offsets"), (perm, (T * k,), "perm"),
                           (inv, (T * k,), "inv"), (status, (1,), "device_status")):
        _need(t, torch.int32, shape, name)
        if t.device != dev:
            raise ValueError(f"{name}: on {t.device}, topk_idx on {dev}")
    _check(_permute_noalloc(_ptr(idx), ctypes.byref(D), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
                            _ptr(status), _stream(stream)), "lmoe_permute_noalloc")
    return counts, offsets, perm, inv, status


def expert_ffn(xq, xs, bank: ExpertBank, offsets, perm, topk_w, k: int, ws=None, stream=None):
    T, d = xq.shape
    D = dims(T, d, bank.E, k, bank.I)
    _need(xq, torch.uint8, (T, d), "xq")
    _need(xs, torch.uint8, (T, d // 32), "xs")
    _need(offsets, torch.int32, (bank.E + 1,), "offsets")
    _need(perm, torch.int32, (T * k,), "perm")
    _need(topk_w, torch.float32, (T, k), "topk_w")
    yp = _empty((T * k, d), torch.float32, xq.device)
    ws = workspace(_ffn_ws(ctypes.byref(D)), xq.device) if ws is None else ws
    W = bank.struct()
    _check(_ffn(_ptr(xq), _ptr(xs), ctypes.byref(W), _ptr(offsets), _ptr(perm), _ptr(topk_w), ctypes.byref(D),
                _ptr(yp), _ptr(ws), ws.numel(), _stream(stream)), "lmoe_expert_ffn")
    return yp, ws


def combine(yp, inv, T: int, k: int, stream=None):
    P, d = yp.shape
    _need(yp, torch.float32, (T * k, d), "yp")
    _need(inv, torch.int32, (T * k,), "inv")
    D = dims(T, d, 32, k, 32)
    y = _empty((T, d), torch.bfloat16, yp.device)
    _check(_combine(_ptr(yp), _ptr(inv), ctypes.byref(D), _ptr(y), _stream(stream)), "lmoe_combine")
    return y


# ---- whole layer -------------------------------------------------------------------

def workspace_size(T: int, d: int, E: int, k: int, I: int) -> int:
    D = dims(T, d, E, k, I)
    return int(_ws_size(ctypes.byref(D)))


class Layer:
    """A LatentMoE layer: router weights (fp32, prepared once into the form the
    router GEMM reads), optional logit bias, expert bank."""

    def __init__(self, Wr: torch.Tensor, bank: ExpertBank, k: int = 16, bias=None, act: int = ACT_MXFP8):
        self.Wr, self.bank, self.k, self.bias, self.act = Wr, bank, k, bias, act
        self.Wr3 = prepare_router(Wr)
        self._ws = None

    def workspace(self, T: int) -> torch.Tensor:
        need = workspace_size(T, self.bank.d, self.bank.E, self.k, self.bank.I)
        if self._ws is None or self._ws.numel() < need:
            self._ws = workspace(need, self.Wr.device)
        return self._ws

    def forward(self, x, y=None, topk_idx=None, topk_w=None, logits=None, stream=None):
        T, d = x.shape
        _need(x, torch.bfloat16, (T, d), "x")
        D = dims(T, d, self.bank.E, self.k, self.bank.I, self.act)
        y = _empty((T, d), torch.bfloat16, x.device) if y is None else y
        ws = self.workspace(T)
        W = self.bank.struct()
        _check(_forward(_ptr(x), _ptr(self.Wr3), _ptr(self.bias), ctypes.byref(W), ctypes.byref(D), _ptr(y),
                        _ptr(topk_idx), _ptr(topk_w), _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)),
               "lmoe_forward")
        return y

    def device_status(self) -> int:
        return last_device_status(self._ws)


def linear_bf16(x, W, out=None, stream=None):
    """out = bf16(x W^T): x bf16 [rows, K], W bf16 [N, K]."""
    rows, K = x.shape
    N = W.shape[0]
    _need(x, torch.bfloat16, (rows, K), "x")
    _need(W, torch.bfloat16, (N, K), "W")
    out = _empty((rows, N), torch.bfloat16, x.device) if out is None else out
    _check(_linear(_ptr(x), _ptr(W), rows, K, N, _ptr(out), _stream(stream)), "lmoe_linear_bf16")
    return out


class Block:
    """hidden -> latent projection, the LatentMoE layer, latent -> hidden."""

    def __init__(self, W_in: torch.Tensor, layer: Layer, W_out: torch.Tensor):
        self.W_in, self.layer, self.W_out = W_in, layer, W_out
        self._ws = None

    def forward(self, x_h, out=None, lat=None, y=None, topk_idx=None, topk_w=None, logits=None, stream=None):
        T, hidden = x_h.shape
        bank, k = self.layer.bank, self.layer.k
        _need(x_h, torch.bfloat16, (T, hidden), "x_h")
        _need(self.W_in, torch.bfloat16, (bank.d, hidden), "W_in")
        _need(self.W_out, torch.bfloat16, (hidden, bank.d), "W_out")
        D = dims(T, bank.d, bank.E, k, bank.I)
        need = int(_block_ws(ctypes.byref(D), hidden))
        if self._ws is None or self._ws.numel() < need:
            self._ws = workspace(need, x_h.device)
        out = _empty((T, hidden), torch.bfloat16, x_h.device) if out is None else out
        W = bank.struct()
        _check(_forward_block(_ptr(x_h), _ptr(self.W_in), _ptr(self.layer.Wr3), _ptr(self.layer.bias), ctypes.byref(W),
                              _ptr(self.W_out), ctypes.byref(D), hidden, _ptr(out), _ptr(lat), _ptr(y), _ptr(topk_idx),
                              _ptr(topk_w), _ptr(logits), _ptr(self._ws), self._ws.numel(), _stream(stream)),
               "lmoe_forward_block")
        return out


def last_device_status(ws) -> int:
    v = _i32()
    _check(_last_status(_ptr(ws), ctypes.byref(v)), "lmoe_last_device_status")
    return int(v.value)
