"""The hidden-width block around the layer: bf16 projections (tensor cores,
fp32 accumulation) and lmoe_forward_block, against the CPU oracle.

Projections are compared element by element: the GPU's fp32 sum and the
oracle's fp64 sum round to the same bf16 except near a rounding boundary or
where the dot product cancels, so every element must be within one bf16 ulp
of the oracle plus the recursive-summation bound K * 2^-24 * sum_c |x_c W_c|
of an fp32 accumulation (and most are exactly equal).  The layer in the
middle is checked teacher-forced on the GPU's own latent rows and logits
(bit-exact routing, outputs within 1e-2 of the row RMS), as in the layer tests.
"""
import numpy as np
import pytest
import torch

import lmoe_inputs as gen
import oracle
from _util import (bf16_to_f64, check_layer_rows, device_bank, envelope_budget, from_dev_bf16, oracle_rows_parallel,
                   quantize_experts_parallel, to_dev_bf16, ulp_flip_budget)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def assert_within_one_bf16_ulp(got_bf16, ref_bf16, x_bf16, W_bf16):
    g, r = bf16_to_f64(got_bf16), bf16_to_f64(ref_bf16)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 1e-30))) - 7)
    K = x_bf16.shape[1]
    acc_bound = K * 2.0 ** -24 * (np.abs(bf16_to_f64(x_bf16)) @ np.abs(bf16_to_f64(W_bf16)).T)
    bad = np.abs(g - r) > ulp * 1.0001 + acc_bound
    assert not bad.any(), f"{bad.sum()} elements beyond one bf16 ulp + the fp32 summation bound"
    return float((got_bf16 == ref_bf16).mean())


@pytest.mark.parametrize("rows,K,N", [(1, 64, 16), (37, 192, 80), (300, 512, 1024), (129, 7168, 256)])
def test_linear_bf16_against_oracle(cuda_lib, rows, K, N):
    lmoe = cuda_lib
    x = gen.normal_bf16(3, rows + K, 0, rows * K, 1.0).reshape(rows, K)
    W = gen.normal_bf16(4, N + K, 0, N * K, 1.0 / np.sqrt(K)).reshape(N, K)
    y = lmoe.linear_bf16(to_dev_bf16(x, DEV), to_dev_bf16(W, DEV))
    torch.cuda.synchronize()
    exact = assert_within_one_bf16_ulp(from_dev_bf16(y), oracle.linear_bf16(x, W), x, W)
    assert exact > 0.97


def _block_case(lmoe, wl, tokens):
    bank = device_bank(wl, DEV)
    bias = gen.router_bias(wl)
    layer = lmoe.Layer(torch.from_numpy(gen.router_f32(wl)).to(DEV), bank, k=wl.k,
                       bias=None if bias is None else torch.from_numpy(bias).to(DEV))
    W_in, W_out = gen.proj_in_bf16(wl), gen.proj_out_bf16(wl)
    blk = lmoe.Block(to_dev_bf16(W_in, DEV), layer, to_dev_bf16(W_out, DEV))
    x_h = gen.hidden_bf16(wl)
    T = wl.T
    lat = torch.empty((T, wl.d), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((T, wl.d), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((T, wl.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    logits = torch.empty((T, wl.E), dtype=torch.float32, device=DEV)
    out = blk.forward(to_dev_bf16(x_h, DEV), lat=lat, y=y, topk_idx=idx, topk_w=w, logits=logits)
    torch.cuda.synchronize()
    lat_h, y_h, out_h = from_dev_bf16(lat), from_dev_bf16(y), from_dev_bf16(out)
    idx_h, w_h, lg_h = idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()
    tok = np.asarray(tokens, np.int32)
    # S0: latent down-projection
    assert_within_one_bf16_ulp(lat_h[tok], oracle.linear_bf16(x_h[tok], W_in), x_h[tok], W_in)
    # routing on the GPU's logits, experts teacher-forced on the GPU's latent rows
    ridx, rw = oracle.topk_softmax(lg_h, wl.k)
    np.testing.assert_array_equal(idx_h, ridx)
    np.testing.assert_allclose(w_h, rw, rtol=1e-6, atol=1e-9)
    ob = quantize_experts_parallel(wl, np.unique(ridx[tok]))
    y64 = oracle_rows_parallel(lat_h, ridx, rw, ob, wl.d, wl.E, wl.I, tok)
    err, n_ulp, n_env = check_layer_rows(y_h[tok], y64, lat_h[tok], ridx[tok], rw[tok], ob, wl.d, wl.I, 1e-2)
    print(f"{wl.name}: {tok.size} rows checked, worst {err.max():.3e} of rms beyond the output rounding; "
          f"{n_ulp} rows over the plain bar by one-ulp output flips only, {n_env} passed through the h envelope")
    assert n_env <= envelope_budget(tok.size)
    assert n_ulp <= ulp_flip_budget(tok.size)
    # S7': up-projection of the GPU's layer output
    assert_within_one_bf16_ulp(out_h[tok], oracle.linear_bf16(y_h[tok], W_out), y_h[tok], W_out)


def test_forward_block_small(cuda_lib):
    wl = gen.custom("block_small", T=24, d=512, I=64, hidden=1024)
    _block_case(cuda_lib, wl, list(range(24)))


def test_forward_block_full_size_sampled(cuda_lib):
    wl = gen.WORKLOADS["block"]
    _block_case(cuda_lib, wl, sorted(set(range(0, wl.T, 1024)) | {1, 4097, 16384, 32766, 32767}))
