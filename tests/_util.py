"""Test helpers: device expert banks from the shared generator, layout
re-arrangements written out from the header's description, error metrics."""
from __future__ import annotations

import numpy as np

import lmoe_inputs as gen


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_dev_bf16(a_u16: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).to(dev).view(torch.bfloat16)


def from_dev_bf16(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def row_rel_err(y_gpu_bf16: np.ndarray, y_ref_bf16: np.ndarray) -> np.ndarray:
    """max_c |y_gpu - y_ref| / rms(y_ref[t, :]) per row."""
    g, r = bf16_to_f64(y_gpu_bf16), bf16_to_f64(y_ref_bf16)
    rms = np.sqrt((r ** 2).mean(1))
    return np.abs(g - r).max(1) / np.maximum(rms, 1e-30)


def canonical_to_tc(q: np.ndarray, s: np.ndarray, nmat: int, rows: int, K: int):
    """Canonical MXFP4 arrays -> the tensor-core layout (include/lmoe.h):
    codes with K padded to a multiple of 128; scales in 512-byte atoms of
    128 rows x 4 blocks, row 32*j + i / block b at byte 16*i + 4*j + b."""
    Kp = -(-K // 128) * 128
    RT, KC = -(-rows // 128), Kp // 128
    q = q.reshape(nmat, rows, K // 2)
    s = s.reshape(nmat, rows, K // 32)
    qt = np.zeros((nmat, rows, Kp // 2), np.uint8)
    qt[:, :, :K // 2] = q
    st = np.zeros((nmat, RT, KC, 512), np.uint8)
    r = np.arange(rows)
    for b in range(K // 32):
        rt, rr = r // 128, r % 128
        off = (rr % 32) * 16 + (rr // 32) * 4 + (b % 4)
        st[:, rt, b // 4, off] = s[:, r, b]
    return qt.reshape(-1), st.reshape(-1)


def device_bank(wl, dev, chunk: int = 32):
    """The expert bank of workload `wl` quantised on the device, generated in
    chunks of experts (load-time conversion, one chunk of fp32 at a time)."""
    import torch
    from top_routing_mxfp4_gb300 import lmoe
    bank = lmoe.ExpertBank(wl.E, wl.d, wl.I, dev)
    for e0 in range(0, wl.E, chunk):
        e1 = min(wl.E, e0 + chunk)
        for which in ("gate", "up", "down"):
            bank.load(which, e0, torch.from_numpy(gen.expert_f32(wl, which, e0, e1)).to(dev))
    torch.cuda.synchronize()
    return bank
