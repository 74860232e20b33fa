"""End-to-end parity of lmoe_forward (through the C ABI) with the CPU oracle.

Routing is compared bit-exactly given the GPU's own fp32 logits (the oracle's
top-k runs on them); the layer output must be within 1e-2 of each row's RMS
(max abs error / rms(y_ref[t])) against the oracle evaluated on the same
routing.  Large workloads compare a sample of tokens.
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


@pytest.fixture(autouse=True)
def tensor_core_path(cuda_lib):
    """These tests cover the tensor-core path at every batch size (the
    small-batch path has its own tests); restored after each test."""
    old = cuda_lib.small_batch_pairs()
    cuda_lib.set_small_batch_pairs(0)
    yield
    cuda_lib.set_small_batch_pairs(old)

_banks = {}


def _bank(wl):
    key = (wl.E, wl.d, wl.I, wl.seed)
    if key not in _banks:
        _banks.clear()
        _banks[key] = device_bank(wl, DEV)
    return _banks[key]


def _run_forward(lmoe, wl, x=None):
    x = gen.x_bf16(wl) if x is None else x
    bias = gen.router_bias(wl)
    layer = lmoe.Layer(torch.from_numpy(gen.router_f32(wl)).to(DEV), _bank(wl), k=wl.k,
                       bias=None if bias is None else torch.from_numpy(bias).to(DEV))
    T = x.shape[0]
    idx = torch.empty((T, wl.k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
    logits = torch.empty((T, wl.E), dtype=torch.float32, device=DEV)
    y = layer.forward(to_dev_bf16(x, DEV), topk_idx=idx, topk_w=w, logits=logits)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    return x, from_dev_bf16(y), idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()


def _check(wl, x, y, idx, w, logits, tokens):
    """Routing bit-exact on the GPU's logits; output rows within the bar.
    Also counts the rows that passed only through the rounding allowances
    (the output's half ulp, the h decision envelope) and holds that count to
    1 % of the rows checked."""
    ridx, rw = oracle.topk_softmax(logits, wl.k)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=1e-6, atol=1e-9)
    tok = np.asarray(sorted(set(int(t) for t in tokens)), np.int32)
    ob = quantize_experts_parallel(wl, np.unique(ridx[tok]))
    y64 = oracle_rows_parallel(x, ridx, rw, ob, wl.d, wl.E, wl.I, tok)
    err, n_ulp, n_env = check_layer_rows(y[tok], y64, x[tok], ridx[tok], rw[tok], ob, wl.d, wl.I, TOL)
    print(f"{wl.name}: {tok.size} rows checked, worst {err.max():.3e} of rms beyond the output rounding; "
          f"{n_ulp} rows over the plain bar by one-ulp output flips only, {n_env} passed through the h envelope")
    assert n_env <= envelope_budget(tok.size), f"{n_env} of {tok.size} rows needed the h decision envelope"
    assert n_ulp <= ulp_flip_budget(tok.size), f"{n_ulp} of {tok.size} rows had one-ulp flips over the bar"
    return err


def test_forward_tiny_all_tokens(cuda_lib):
    wl = gen.WORKLOADS["tiny"]
    x, y, idx, w, lg = _run_forward(cuda_lib, wl)
    _check(wl, x, y, idx, w, lg, list(range(wl.T)))


def test_forward_decode_all_tokens(cuda_lib):
    wl = gen.WORKLOADS["decode"]
    x, y, idx, w, lg = _run_forward(cuda_lib, wl)
    _check(wl, x, y, idx, w, lg, list(range(wl.T)))


@pytest.mark.parametrize("name", ["prefill", "skewed"])
def test_forward_prefill_sampled(cuda_lib, name):
    wl = gen.WORKLOADS[name]
    x, y, idx, w, lg = _run_forward(cuda_lib, wl)
    # every 128th token across the batch (first and last included), and every
    # token of the hottest expert's first 96-token tile (its first 96 tokens
    # in id order, which the expert GEMMs process as one tile)
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    hot = int(np.argmax(counts))
    hot_tokens = np.flatnonzero((idx == hot).any(1))[:96]
    toks = sorted(set(range(0, wl.T, 128)) | {wl.T - 1} | set(int(t) for t in hot_tokens))
    assert len(toks) >= 150
    _check(wl, x, y, idx, w, lg, toks)
    if name == "skewed":
        assert counts.max() / counts.mean() > 5.0


@pytest.mark.parametrize("T", [1, 3, 131])
def test_forward_ragged_token_counts(cuda_lib, T):
    wl = gen.custom(f"ragged{T}", T=T, d=512, I=64)
    x, y, idx, w, lg = _run_forward(cuda_lib, wl)
    _check(wl, x, y, idx, w, lg, sorted(set([0, T // 2, T - 1])))


def test_forward_ragged_shapes(cuda_lib):
    wl = gen.custom("oddshape", T=45, d=384, I=160, E=70, k=7)
    x, y, idx, w, lg = _run_forward(cuda_lib, wl)
    _check(wl, x, y, idx, w, lg, list(range(0, 45, 4)))


@pytest.mark.parametrize("T,E,k", [(64, 256, 32), (64, 896, 1), (17, 130, 9)])
def test_forward_small_batch_routing_edges(cuda_lib, T, E, k):
    """Batches the routing kernel permutes itself (up to 64 tokens): every
    token's bit of the 64-bit masks in use (T = 64), the largest k (more
    selections than warps: the selection's fall-back rounds), k = 1, and an
    expert count that is not a multiple of 32."""
    wl = gen.custom(f"route_edge_{T}_{E}_{k}", T=T, d=512, I=64, E=E, k=k)
    x, y, idx, w, lg = _run_forward(cuda_lib, wl)
    _check(wl, x, y, idx, w, lg, sorted(set([0, 1, T // 2, T - 1])))


@pytest.mark.parametrize("d,I,k", [(3584, 512, 19), (3584, 512, 20), (1408, 160, 16), (256, 512, 16),
                                   (128, 512, 16)])
def test_forward_split_k_gateup(cuda_lib, d, I, k):
    """Batch 1 with at most half as many gate/up work items as SMs: each item
    runs as two K halves on two SMs and the later half forms h from the sum
    of both halves' fp32 accumulators.  Cases: 19 experts x 4 weight tiles =
    76 items (the most that split on 152 SMs) and 80 (the first that do
    not), 11 K chunks (halves of 5 and 6) with I = 160 (three of the second
    weight tile's four epilogue warps hold no rows of I), one K chunk per
    half (d = 256), and one K chunk in all (d = 128: no split).  The
    arrival counters show which items split; the output is checked against
    the oracle and repeated bit for bit."""
    lmoe = cuda_lib
    wl = gen.custom(f"ksplit_{d}_{I}_{k}", T=1, d=d, I=I, E=64, k=k)
    layer = lmoe.Layer(torch.from_numpy(gen.router_f32(wl)).to(DEV), _bank(wl), k=k)
    v = lmoe.forward_workspace_views(1, d, wl.E, k, I)
    assert v.path == 0 and v.tile_tokens == 16 and v.ksplit >= 0
    x = gen.x_bf16(wl)
    idx = torch.empty((1, k), dtype=torch.int32, device=DEV)
    w = torch.empty((1, k), dtype=torch.float32, device=DEV)
    logits = torch.empty((1, wl.E), dtype=torch.float32, device=DEV)
    ys = []
    for _ in range(2):
        y = layer.forward(to_dev_bf16(x, DEV), topk_idx=idx, topk_w=w, logits=logits)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        ys.append(from_dev_bf16(y))
    assert np.array_equal(ys[0], ys[1])
    MT = -(-I // 128)
    n_items = k * MT  # one token tile per selected expert
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    split = 2 * n_items <= sms and n_items <= 128 and d // 128 >= 2
    cnt = layer._ws[v.ksplit:v.ksplit + 128 * 16].view(torch.int32).view(128, 4)[:n_items].cpu().numpy()
    m = np.arange(n_items)[:, None] % MT
    has_rows = 128 * m + 32 * np.arange(4)[None, :] < I
    np.testing.assert_array_equal(cnt, np.where(has_rows & split, 2, 0))
    _check(wl, x, ys[0], idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy(), [0])


def _token_tile(wl):
    """Token tile the library picks for a batch (by the mean pairs per expert)."""
    return 16 if wl.P <= 4 * wl.E else 32 if wl.P <= 16 * wl.E else 96


@pytest.mark.parametrize("T,E,k", [(600, 24, 4), (301, 15, 6), (600, 8, 4), (301, 10, 6)])
def test_forward_fused_combine_all_tokens(cuda_lib, T, E, k):
    """Batches with more than 16 routed pairs per expert use 96-token tiles,
    and the down GEMM's epilogue adds each pair's weighted output straight
    into its token's fp32 row (fp32 atomics; the k terms in an unspecified
    order).  Every token is checked: one to four ragged token tiles per
    expert, d = 3 weight tiles, I = 160 (a ragged last K chunk)."""
    wl = gen.custom(f"fused{T}_{E}", T=T, d=384, I=160, E=E, k=k)
    assert wl.P > 16 * wl.E
    x, y, idx, w, lg = _run_forward(cuda_lib, wl)
    _check(wl, x, y, idx, w, lg, list(range(T)))
    assert np.bincount(idx.ravel(), minlength=E).max() > _token_tile(wl)  # experts span several token tiles
    # a zero batch accumulates to exactly zero
    _, y0, _, _, _ = _run_forward(cuda_lib, wl, np.zeros((T, wl.d), np.uint16))
    assert np.all((y0 & 0x7FFF) == 0)


@pytest.mark.parametrize("d,E", [(256, 12), (128, 6)])
def test_forward_fused_combine_single_weight_band(cuda_lib, d, E):
    """Fused path whose down GEMM has one item per token tile (two 128-row
    weight tiles per item: d = 256, or d = 128 where the item's second tile
    is a copy the epilogue drops), so the second output-column band is empty;
    every token checked."""
    wl = gen.custom(f"fused_d{d}", T=300, d=d, I=96, E=E, k=4)
    assert _token_tile(wl) == 96
    x, y, idx, w, lg = _run_forward(cuda_lib, wl)
    _check(wl, x, y, idx, w, lg, list(range(wl.T)))


def test_forward_32_token_tiles_all_experts(cuda_lib):
    """Between 4 and 16 pairs per expert (T = 512 over 896 experts): 32-token
    tiles, two weight tiles per down stage, per-pair outputs and the
    slot-order combine."""
    wl = gen.custom("mid512", T=512, d=512, I=64)
    assert 4 * wl.E < wl.P <= 16 * wl.E
    x, y, idx, w, lg = _run_forward(cuda_lib, wl)
    _check(wl, x, y, idx, w, lg, [0, 1, 100, 255, 256, 400, 511])


def test_forward_zero_input_gives_zero(cuda_lib):
    wl = gen.WORKLOADS["tiny"]
    x = np.zeros((4, wl.d), np.uint16)
    _, y, _, _, _ = _run_forward(cuda_lib, wl, x)
    assert np.all((y & 0x7FFF) == 0)


def test_forward_empty_batch_is_noop(cuda_lib):
    lmoe = cuda_lib
    wl = gen.WORKLOADS["tiny"]
    layer = lmoe.Layer(torch.from_numpy(gen.router_f32(wl)).to(DEV), _bank(wl), k=wl.k)
    y = layer.forward(torch.empty((0, wl.d), dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert y.shape == (0, wl.d)


def test_fused_combine_run_to_run_difference_is_bounded(cuda_lib):
    """Large batches sum each token's k pair outputs with fp32 atomics in an
    unspecified order, so two runs may differ in the last fp32 bits before the
    bf16 rounding: at most one bf16 ulp per element, in few elements.  Small
    batches (slot-order combine) must be bit-identical."""
    lmoe = cuda_lib
    wl = gen.custom("rerun600", T=600, d=384, I=160, E=24, k=4)
    x = gen.x_bf16(wl)
    outs = [_run_forward(lmoe, wl, x)[1] for _ in range(3)]
    from _util import bf16_to_f64, half_ulp_bf16
    y0 = bf16_to_f64(outs[0])
    for y in outs[1:]:
        y1 = bf16_to_f64(y)
        ulp = 2 * half_ulp_bf16(np.maximum(np.abs(y0), np.abs(y1)))
        assert np.all(np.abs(y0 - y1) <= ulp), "outputs differ by more than one bf16 ulp between runs"
        frac = (y0 != y1).mean()
        print(f"fused combine: {frac:.2e} of outputs differ by one ulp between runs")
        assert frac < 1e-3
    wl_s = gen.custom("rerun64", T=64, d=512, I=64)
    xs = gen.x_bf16(wl_s)
    ys = [_run_forward(lmoe, wl_s, xs)[1] for _ in range(2)]
    np.testing.assert_array_equal(ys[0], ys[1])
