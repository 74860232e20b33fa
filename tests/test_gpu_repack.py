"""Load-time conversion of an MXFP4 checkpoint into the expert GEMMs' layout
(lmoe_repack_mxfp4) and the per-matrix distribution of its E8M0 scales
(lmoe_mxfp4_scale_histogram), through the C ABI.

The checkpoint is the oracle's MXFP4 quantisation of the generator's fp32
weights (canonical bytes).  The repacked bank must equal, byte for byte,
(a) the same bytes rearranged in numpy from the header's description of the
layout, and (b) the bank the device quantiser writes from the fp32 weights
directly.  The histograms must equal numpy's counts of the oracle's scale
bytes.  Whole banks of both expert shapes are streamed through one staging
buffer of a few experts, as a loader would do layer by layer.
"""
import numpy as np
import pytest
import torch

import lmoe_inputs as gen
from _util import canonical_to_tc, device_bank, quantize_experts_parallel

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("nmat,rows,K", [(3, 160, 96), (2, 300, 544), (1, 128, 128), (5, 512, 3584)])
def test_repack_matches_layout_description(cuda_lib, nmat, rows, K):
    lmoe = cuda_lib
    rng = np.random.default_rng(nmat * rows + K)
    q = rng.integers(0, 256, size=(nmat, rows, K // 2), dtype=np.uint8)
    s = rng.integers(100, 140, size=(nmat, rows, K // 32), dtype=np.uint8)
    qt_ref, st_ref = canonical_to_tc(q, s, nmat, rows, K)
    # destinations start as garbage: padding must be written, not assumed
    qb, sb = lmoe.mxfp4_bytes(nmat, rows, K, lmoe.LAYOUT_TC)
    q_tc = torch.full((qb,), 0xA5, dtype=torch.uint8, device=DEV)
    s_tc = torch.full((sb,), 0x5A, dtype=torch.uint8, device=DEV)
    lmoe.repack_mxfp4(torch.from_numpy(q).to(DEV), torch.from_numpy(s).to(DEV), nmat, rows, K, q_tc, s_tc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q_tc.cpu().numpy(), qt_ref)
    np.testing.assert_array_equal(s_tc.cpu().numpy(), st_ref)
    for layout, arr in ((lmoe.LAYOUT_CANONICAL, torch.from_numpy(s).to(DEV)), (lmoe.LAYOUT_TC, s_tc)):
        h = lmoe.scale_histogram(arr, nmat, rows, K, layout).cpu().numpy()
        ref = np.stack([np.bincount(s[m].ravel(), minlength=256) for m in range(nmat)])
        np.testing.assert_array_equal(h, ref)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_checkpoint_streamed_into_bank_equals_device_quantiser(cuda_lib, name):
    """Every expert of the workload's bank: oracle-quantised canonical bytes
    streamed through a staging buffer of 16 experts into an ExpertBank equal
    the device-quantised bank byte for byte; the bank's scale histograms
    equal numpy's counts of the oracle's scales."""
    lmoe = cuda_lib
    wl = gen.WORKLOADS[name]
    E, d, I = wl.E, wl.d, wl.I
    ob = quantize_experts_parallel(wl, range(E))
    gq, gs, uq, us, dq, ds = ob.arrays
    canon = {"gate": (gq.reshape(E, I, d // 2), gs.reshape(E, I, d // 32)),
             "up": (uq.reshape(E, I, d // 2), us.reshape(E, I, d // 32)),
             "down": (dq.reshape(E, d, I // 2), ds.reshape(E, d, I // 32))}
    bank = lmoe.ExpertBank(E, d, I, DEV)
    for t in (bank.gate_q, bank.gate_s, bank.up_q, bank.up_s, bank.down_q, bank.down_s):
        t.fill_(0x77)
    chunk = 16
    for which, (q, s) in canon.items():
        stage_q = torch.empty((chunk,) + q.shape[1:], dtype=torch.uint8, device=DEV)
        stage_s = torch.empty((chunk,) + s.shape[1:], dtype=torch.uint8, device=DEV)
        for e0 in range(0, E, chunk):
            n = min(chunk, E - e0)
            stage_q[:n].copy_(torch.from_numpy(q[e0:e0 + n]))
            stage_s[:n].copy_(torch.from_numpy(s[e0:e0 + n]))
            bank.load_mxfp4(which, e0, stage_q[:n], stage_s[:n])
            torch.cuda.synchronize()  # the staging buffer is refilled next
    ref = device_bank(wl, DEV)
    for a in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        assert torch.equal(getattr(bank, a), getattr(ref, a)), a
    hist = bank.scale_histograms()
    for which, (q, s) in canon.items():
        want = np.stack([np.bincount(s[e].ravel(), minlength=256) for e in range(E)])
        np.testing.assert_array_equal(hist[which].cpu().numpy(), want)
