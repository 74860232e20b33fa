"""The small-batch path of lmoe_forward (batch-1 to 16-token decode steps:
three weight-streaming kernels) against the CPU oracle, through the C ABI.

Same checks as the tensor-core path: routing bit-exact given the GPU's own
logits, logits within 1e-4 of the row RMS of the oracle's, every token's
output within 1e-2 of its row RMS (with the one-ulp / h-envelope counts held
to their budgets), and both MXFP8 roundings bit for bit (x per token, h per
pair, read back from the workspace).  Also: results are bit-identical run to
run, the workspace's counter is left ready for the next call, and the
tensor-core path gives the same routing on the same batch.
"""
import numpy as np
import pytest
import torch

import lmoe_inputs as gen
import oracle
from _util import (check_layer_rows, device_bank, envelope_budget, from_dev_bf16, oracle_rows_parallel,
                   quantize_experts_parallel, to_dev_bf16, ulp_flip_budget)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-2

_banks = {}


def _bank(wl):
    key = (wl.E, wl.d, wl.I, wl.seed)
    if key not in _banks:
        _banks.clear()
        _banks[key] = device_bank(wl, DEV)
    return _banks[key]


@pytest.fixture
def small_path(cuda_lib):
    """Every batch of up to 256 pairs takes the small-batch path; restored after."""
    old = cuda_lib.small_batch_pairs()
    cuda_lib.set_small_batch_pairs(256)
    yield cuda_lib
    cuda_lib.set_small_batch_pairs(old)


def _forward(lmoe, wl, x, hcap=False, act=None):
    bias = gen.router_bias(wl)
    layer = lmoe.Layer(torch.from_numpy(gen.router_f32(wl)).to(DEV), _bank(wl), k=wl.k,
                       bias=None if bias is None else torch.from_numpy(bias).to(DEV),
                       act=lmoe.ACT_MXFP8 if act is None else act)
    T = x.shape[0]
    idx = torch.empty((T, wl.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    logits = torch.empty((T, wl.E), dtype=torch.float32, device=DEV)
    cap = None
    if hcap:
        cap = torch.full((T * wl.k * wl.I,), float("nan"), dtype=torch.float32, device=DEV)
        lmoe.set_h_capture(cap)
    try:
        y = layer.forward(to_dev_bf16(x, DEV), topk_idx=idx, topk_w=w, logits=logits)
        torch.cuda.synchronize()
    finally:
        if hcap:
            lmoe.set_h_capture(None)
    assert layer.device_status() == 0
    return layer, from_dev_bf16(y), idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy(), cap


def _check_all(lmoe, wl, x, y, idx, w, lg):
    ref_lg = oracle.router_logits(x, gen.router_f32(wl), gen.router_bias(wl))
    rms = np.sqrt((ref_lg.astype(np.float64) ** 2).mean(1, keepdims=True))
    assert (np.abs(lg - ref_lg) / rms).max() < 1e-4
    ridx, rw = oracle.topk_softmax(lg, wl.k)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=1e-6, atol=1e-9)
    tok = np.arange(wl.T, dtype=np.int32)
    ob = quantize_experts_parallel(wl, np.unique(ridx))
    y64 = oracle_rows_parallel(x, ridx, rw, ob, wl.d, wl.E, wl.I, tok)
    err, n_ulp, n_env = check_layer_rows(y, y64, x, ridx, rw, ob, wl.d, wl.I, TOL)
    print(f"{wl.name} (small path): {wl.T} rows, worst {err.max():.3e} of rms beyond the output rounding; "
          f"{n_ulp} one-ulp rows, {n_env} envelope rows")
    assert n_env <= envelope_budget(wl.T) and n_ulp <= ulp_flip_budget(wl.T)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_small_path_decode_shape_all_tokens(small_path, T):
    lmoe = small_path
    wl = gen.custom(f"small{T}", T=T, d=3584, I=512)
    v = lmoe.forward_workspace_views(T, wl.d, wl.E, wl.k, wl.I)
    assert v.path == 1 and lmoe.forward_kernel_count(T, wl.d, wl.E, wl.k, wl.I) == 3
    x = gen.x_bf16(wl)
    layer, y, idx, w, lg, cap = _forward(lmoe, wl, x, hcap=True)
    _check_all(lmoe, wl, x, y, idx, w, lg)
    # MXFP8 of x (rows = tokens) and of h (rows = pairs), bit for bit
    ws = layer._ws
    P, d, I = T * wl.k, wl.d, wl.I

    def atoms(base, rows, nb):
        KC = -(-nb // 4)
        r = np.arange(rows)[:, None]
        b = np.arange(nb)[None, :]
        off = ((r >> 7) * KC + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3)
        return ws[base:base + int(off.max()) + 1].cpu().numpy()[off]

    rq, rs = oracle.quant_mxfp8(x)
    np.testing.assert_array_equal(ws[v.xq:v.xq + T * d].cpu().numpy().reshape(T, d), rq)
    np.testing.assert_array_equal(atoms(v.xs, T, d // 32), rs)
    h = cap.view(P, I).cpu().numpy().astype(np.float64)
    assert np.isfinite(h).all()
    hrq, hrs = oracle.quant_mxfp8_f64(h)
    np.testing.assert_array_equal(ws[v.hq:v.hq + P * I].cpu().numpy().reshape(P, I), hrq)
    np.testing.assert_array_equal(atoms(v.hs, P, I // 32), hrs)
    # deterministic, and the routing kernel's counter was left at zero for the next call
    _, y2, idx2, _, lg2, _ = _forward(lmoe, wl, x)
    np.testing.assert_array_equal(y2, y)
    np.testing.assert_array_equal(lg2, lg)


@pytest.mark.parametrize("name,T,d,I,E,k", [("sm_odd", 5, 384, 160, 70, 7), ("sm_tiny", 8, 512, 64, 896, 16),
                                            ("sm_wide", 3, 512, 96, 1536, 8), ("sm_k32", 4, 256, 64, 64, 32)])
def test_small_path_ragged_shapes(small_path, name, T, d, I, E, k):
    lmoe = small_path
    wl = gen.custom(name, T=T, d=d, I=I, E=E, k=k)
    assert lmoe.forward_workspace_views(T, d, E, k, I).path == 1
    x = gen.x_bf16(wl)
    _, y, idx, w, lg, _ = _forward(lmoe, wl, x)
    _check_all(lmoe, wl, x, y, idx, w, lg)


def test_small_path_skewed_router_bias_and_zero_input(small_path):
    lmoe = small_path
    wl = gen.custom("sm_skew", T=6, d=3584, I=512, zipf_s=1.2, zipf_beta=0.18)
    x = gen.x_bf16(wl)
    _, y, idx, w, lg, _ = _forward(lmoe, wl, x)
    _check_all(lmoe, wl, x, y, idx, w, lg)
    _, y0, _, _, _, _ = _forward(lmoe, wl, np.zeros((3, wl.d), np.uint16))
    assert np.all((y0 & 0x7FFF) == 0)


def test_small_and_tensor_core_paths_agree(small_path):
    """The same batch through both paths: identical routing (their logits
    differ only in fp32 summation order, far below any gap between the 16th
    and 17th logit here), outputs within the bar of each other."""
    lmoe = small_path
    wl = gen.custom("sm_vs_tc", T=8, d=3584, I=512)
    x = gen.x_bf16(wl)
    _, ys, idxs, ws_, lgs, _ = _forward(lmoe, wl, x)
    lmoe.set_small_batch_pairs(0)
    assert lmoe.forward_workspace_views(wl.T, wl.d, wl.E, wl.k, wl.I).path == 0
    _, yt, idxt, wt, lgt, _ = _forward(lmoe, wl, x)
    np.testing.assert_array_equal(idxs, idxt)
    rms = np.sqrt((lgt.astype(np.float64) ** 2).mean(1, keepdims=True))
    assert (np.abs(lgs - lgt) / rms).max() < 1e-5
    from _util import bf16_to_f64
    a, b = bf16_to_f64(ys), bf16_to_f64(yt)
    assert (np.abs(a - b).max(1) / np.sqrt((b ** 2).mean(1))).max() < TOL


@pytest.mark.parametrize("T", [1, 2, 8])
def test_default_path_decode_shape_all_tokens(cuda_lib, T):
    """The library's default choice of path at one, two and eight tokens (the
    tensor-core path with its fused expert kernel, since the small-batch
    path is opt-in), every token against the oracle."""
    lmoe = cuda_lib
    assert lmoe.small_batch_pairs() == lmoe.SMALL_BATCH_PAIRS_DEFAULT == 0
    wl = gen.custom(f"dflt{T}", T=T, d=3584, I=512)
    assert lmoe.forward_workspace_views(T, wl.d, wl.E, wl.k, wl.I).path == 0
    x = gen.x_bf16(wl)
    _, y, idx, w, lg, _ = _forward(lmoe, wl, x)
    _check_all(lmoe, wl, x, y, idx, w, lg)
    # deterministic run to run (the combine sums each token's pairs in slot order)
    _, y2, _, _, _, _ = _forward(lmoe, wl, x)
    np.testing.assert_array_equal(y2, y)


def test_sixteen_token_step_all_tokens_default_path(cuda_lib):
    """A 16-token decode step (256 pairs) with the library's default choice of
    path, every token against the oracle."""
    lmoe = cuda_lib
    wl = gen.custom("step16", T=16, d=3584, I=512)
    x = gen.x_bf16(wl)
    _, y, idx, w, lg, _ = _forward(lmoe, wl, x)
    _check_all(lmoe, wl, x, y, idx, w, lg)


@pytest.mark.parametrize("T", [1, 2, 8])
def test_small_path_fp4_activations_all_tokens(small_path, T):
    """The full-FP4 variant (x and h rounded to MXFP4) against the oracle's
    FP4 mode: routing as before, every token within the bar (after the
    output's own bf16 rounding), and both MXFP4 roundings bit for bit."""
    lmoe = small_path
    wl = gen.custom(f"fp4_{T}", T=T, d=3584, I=512)
    d, I, k = wl.d, wl.I, wl.k
    x = gen.x_bf16(wl)
    layer, y, idx, w, lg, cap = _forward(lmoe, wl, x, hcap=True, act=lmoe.ACT_MXFP4)
    ridx, rw = oracle.topk_softmax(lg, k)
    np.testing.assert_array_equal(idx, ridx)
    ob = quantize_experts_parallel(wl, np.unique(ridx))
    _, y64 = oracle.moe_tokens(x, ridx, rw, ob, d, wl.E, I, want_f64=True, act=oracle.ACT_MXFP4)
    from _util import bf16_to_f64, half_ulp_bf16
    g = bf16_to_f64(y)
    rms = np.sqrt((y64 ** 2).mean(1))
    err = (np.maximum(np.abs(g - y64) - half_ulp_bf16(g), 0.0).max(1)) / rms
    print(f"fp4_{T}: worst {err.max():.3e} of rms beyond the output rounding")
    assert err.max() <= TOL
    v = lmoe.forward_workspace_views(T, d, wl.E, k, I)
    ws = layer._ws
    P = T * k

    def atoms(base, rows, nb):
        KC = -(-nb // 4)
        r = np.arange(rows)[:, None]
        b = np.arange(nb)[None, :]
        off = ((r >> 7) * KC + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3)
        return ws[base:base + int(off.max()) + 1].cpu().numpy()[off]

    rq, rs = oracle.quant_mxfp4_f64(bf16_to_f64(x))
    np.testing.assert_array_equal(ws[v.xq:v.xq + T * d // 2].cpu().numpy().reshape(T, d // 2), rq)
    np.testing.assert_array_equal(atoms(v.xs, T, d // 32), rs)
    h = cap.view(P, I).cpu().numpy().astype(np.float64)
    hrq, hrs = oracle.quant_mxfp4_f64(h)
    np.testing.assert_array_equal(ws[v.hq:v.hq + P * I // 2].cpu().numpy().reshape(P, I // 2), hrq)
    np.testing.assert_array_equal(atoms(v.hs, P, I // 32), hrs)


def test_fp4_activations_refused_on_the_tensor_core_path(cuda_lib):
    lmoe = cuda_lib
    wl = gen.custom("fp4_tc", T=8, d=512, I=64)
    old = lmoe.small_batch_pairs()
    lmoe.set_small_batch_pairs(0)
    try:
        with pytest.raises(lmoe.LmoeError) as ei:
            _forward(lmoe, wl, gen.x_bf16(wl), act=lmoe.ACT_MXFP4)
        assert ei.value.code == lmoe.ERR_UNSUPPORTED
    finally:
        lmoe.set_small_batch_pairs(old)
