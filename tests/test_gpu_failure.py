"""The expert GEMMs' failure path, without a GPU fault.

Every mbarrier wait in the expert GEMMs is bounded: when it runs out the
kernel records LMOE_ERR_TIMEOUT in the workspace's status word, all roles
leave their loops (an MMA issuer first waits, bounded, for its MMAs in
flight), tensor memory is freed and the kernel returns.  Here the
test-only hook lmoe_set_wait_test makes the first pipeline stage of every
CTA never fill (no copy is issued for it, nothing else changes) with a
10-millisecond limit, so those waits run out; the host reads the status,
and the same context then runs the layer correctly.
"""
import numpy as np
import pytest
import torch

import lmoe_inputs as gen
import oracle
from _util import device_bank, from_dev_bf16, to_dev_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_expert_gemm_wait_runs_out_and_reports_timeout(cuda_lib):
    lmoe = cuda_lib
    wl = gen.WORKLOADS["tiny"]
    old = lmoe.small_batch_pairs()
    lmoe.set_small_batch_pairs(0)  # the tensor-core path, whose GEMMs have the bounded waits
    try:
        bank = device_bank(wl, DEV)
        layer = lmoe.Layer(torch.from_numpy(gen.router_f32(wl)).to(DEV), bank, k=wl.k)
        x = gen.x_bf16(wl)
        xd = to_dev_bf16(x, DEV)
        lmoe.set_wait_test(True, 20_000_000)  # about 10 ms of SM clocks at 2 GHz
        try:
            layer.forward(xd)
            torch.cuda.synchronize()
        finally:
            lmoe.set_wait_test(False, 0)
        assert layer.device_status() == lmoe.ERR_TIMEOUT
        # the context is still usable: the next call is clean and correct
        idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device=DEV)
        w = torch.empty((wl.T, wl.k), dtype=torch.float32, device=DEV)
        lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device=DEV)
        y = layer.forward(xd, topk_idx=idx, topk_w=w, logits=lg)
        torch.cuda.synchronize()
        assert layer.device_status() == lmoe.OK
        ridx, rw = oracle.topk_softmax(lg.cpu().numpy(), wl.k)
        np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
        ob = oracle.quantize_experts(wl, experts=np.unique(ridx))
        yref = oracle.moe_tokens(x, ridx, rw, ob, wl.d, wl.E, wl.I)
        f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        yg, yr = f(from_dev_bf16(y)), f(yref)
        assert (np.abs(yg - yr).max(1) / np.sqrt((yr ** 2).mean(1))).max() <= 1e-2
    finally:
        lmoe.set_small_batch_pairs(old)


def test_wait_test_hook_rejects_a_stall_without_a_limit(cuda_lib):
    with pytest.raises(cuda_lib.LmoeError):
        cuda_lib.set_wait_test(True, 0)
