"""Every MXFP8 quantisation on lmoe_forward's path, bit for bit.

The layer rounds two activations to MXFP8 before the tensor cores read them
(e4m3 codes, one E8M0 scale per 32 elements): the latent x of every routed
pair, written by the activation scatter into the expert GEMM's tiled token
rows, and the gated product h = silu(g) * u, rounded in the gate/up GEMM's
epilogue.  Both are read back from the forward's workspace (its layout comes
from lmoe_forward_workspace_views) and compared, every code and every scale
byte of every routed pair, with the oracle's quantisation of the same
values: the bf16 x of the pair's token, and the fp32 h the epilogue rounded
(captured with lmoe_set_h_capture).  The three batch sizes run the three
token-tile shapes of the expert GEMMs (16, 32 and 96 tokens per tile), whose
epilogues store h differently.
"""
import numpy as np
import pytest
import torch

import lmoe_inputs as gen
import oracle
from _util import device_bank, to_dev_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

_bank = {}


def _get_bank(wl):
    key = (wl.E, wl.d, wl.I, wl.seed)
    if key not in _bank:
        _bank.clear()
        _bank[key] = device_bank(wl, DEV)
    return _bank[key]


def atom_scales(atoms: torch.Tensor, R: torch.Tensor, nblocks: int, tile: int) -> np.ndarray:
    """Scale bytes [len(R), nblocks] of token rows R from the tiled layout:
    row rr = R % tile of tile R // tile, block b at byte
    (tile_index * KC + b / 4) * 512 + 16 (rr % 32) + 4 (rr / 32) + b % 4,
    KC = ceil(nblocks / 4)."""
    KC = -(-nblocks // 4)
    b = torch.arange(nblocks, device=R.device, dtype=torch.int64)[None, :]
    r = R.to(torch.int64)[:, None]
    ti, rr = r // tile, r % tile
    off = (ti * KC + (b >> 2)) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (b & 3)
    return atoms[off].cpu().numpy()


@pytest.fixture(autouse=True)
def tensor_core_path(cuda_lib):
    """These checks cover the tensor-core path (the small-batch path has its
    own bit-exact checks); restored after each test."""
    old = cuda_lib.small_batch_pairs()
    cuda_lib.set_small_batch_pairs(0)
    yield
    cuda_lib.set_small_batch_pairs(old)


@pytest.mark.parametrize("T,tile", [(1, 16), (2, 16), (64, 16), (512, 32), (2048, 96)])
def test_forward_mxfp8_operands_bit_exact(cuda_lib, T, tile):
    lmoe = cuda_lib
    wl = gen.custom(f"mxfp8_exact_{T}", T=T, d=3584, I=512)
    d, I, k, E = wl.d, wl.I, wl.k, wl.E
    bank = _get_bank(wl)
    layer = lmoe.Layer(torch.from_numpy(gen.router_f32(wl)).to(DEV), bank, k=k)
    v = lmoe.forward_workspace_views(T, d, E, k, I)
    assert v.tile_tokens == tile
    x = gen.x_bf16(wl)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    hcap = torch.full((v.rows * I,), float("nan"), dtype=torch.float32, device=DEV)
    lmoe.set_h_capture(hcap)
    try:
        layer.forward(to_dev_bf16(x, DEV), topk_idx=idx)
        torch.cuda.synchronize()
    finally:
        lmoe.set_h_capture(None)
    assert layer.device_status() == 0
    ws = layer._ws
    P = T * k
    R = ws[v.dst_row:v.dst_row + 4 * P].view(torch.int32).to(torch.int64)  # atom rows (scale factors)
    Q = ws[v.code_row:v.code_row + 4 * P].view(torch.int32).to(torch.int64)  # code rows (permuted order)
    Rh, Qh = R.cpu().numpy(), Q.cpu().numpy()
    assert Rh.min() >= 0 and np.unique(Rh).size == P
    assert np.array_equal(np.sort(Qh), np.arange(P)) and v.rows == P + v.tile_tokens
    # x: every routed pair's code row holds MXFP8(x[t]) of its token t = p / k
    xq = ws[v.xq:v.xq + v.rows * d].view(v.rows, d)[Q].cpu().numpy()
    xs = atom_scales(ws[v.xs:v.hq], R, d // 32, v.tile_tokens)
    rq, rs = oracle.quant_mxfp8(x)
    tok = np.arange(P) // k
    bad = np.nonzero((xq != rq[tok]).any(1) | (xs != rs[tok]).any(1))[0]
    assert bad.size == 0, f"{bad.size} of {P} pairs' x rows differ from the oracle (first pair {bad[:1]})"
    # h: every pair's codes and scales equal the oracle's rounding of the fp32 h the GEMM produced
    h = hcap.view(v.rows, I)[Q].cpu().numpy().astype(np.float64)
    assert np.isfinite(h).all(), "the epilogue did not capture h for every routed pair"
    hq = ws[v.hq:v.hq + v.rows * I].view(v.rows, I)[Q].cpu().numpy()
    hs = atom_scales(ws[v.hs:], R, I // 32, v.tile_tokens)
    hrq, hrs = oracle.quant_mxfp8_f64(h)
    bad_q = np.nonzero((hq != hrq).any(1))[0]
    bad_s = np.nonzero((hs != hrs).any(1))[0]
    assert bad_q.size == 0 and bad_s.size == 0, (f"h of {bad_q.size} pairs (codes) / {bad_s.size} pairs (scales) of "
                                                 f"{P} differ from the oracle's MXFP8 of the same fp32 values")
    print(f"T={T}: {P} pairs, x {P * d} codes + {P * d // 32} scales, h {P * I} codes + {P * I // 32} scales "
          f"bit-exact")


@pytest.mark.parametrize("T,skew", [(1, False), (64, False), (64, True)])
def test_forward_permute_matches_oracle(cuda_lib, T, skew):
    """The forward's permute of a small batch (done inside the routing kernel
    from per-expert token masks): every pair's code row is the oracle's
    stable counting-sort position, and its scale-atom row follows from the
    oracle's counts, offsets and the token tile.  Skewed routing puts more
    than one token tile's worth of pairs on some experts."""
    lmoe = cuda_lib
    kw = dict(zipf_s=1.2, zipf_beta=0.5) if skew else {}  # skewed: up to 50 pairs on one expert
    wl = gen.custom(f"perm_small_{T}_{int(skew)}", T=T, d=3584, I=512, **kw)
    d, I, k, E = wl.d, wl.I, wl.k, wl.E
    bank = _get_bank(wl)
    bias = gen.router_bias(wl)
    layer = lmoe.Layer(torch.from_numpy(gen.router_f32(wl)).to(DEV), bank, k=k,
                       bias=None if bias is None else torch.from_numpy(bias).to(DEV))
    v = lmoe.forward_workspace_views(T, d, E, k, I)
    x = gen.x_bf16(wl)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    y1 = layer.forward(to_dev_bf16(x, DEV), topk_idx=idx).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    ih = idx.cpu().numpy()
    counts, offsets, perm, inv = oracle.permute(ih, E)
    P, NT = T * k, v.tile_tokens
    ws = layer._ws
    Q = ws[v.code_row:v.code_row + 4 * P].view(torch.int32).cpu().numpy()
    R = ws[v.dst_row:v.dst_row + 4 * P].view(torch.int32).cpu().numpy()
    np.testing.assert_array_equal(Q, inv)
    tiles = (counts.astype(np.int64) + NT - 1) // NT
    pad = np.concatenate([[0], np.cumsum(tiles)[:-1]]) * NT  # first atom row of each expert's tiles
    e = ih.reshape(-1)
    np.testing.assert_array_equal(R, pad[e] + (inv - offsets[e]))
    if skew:
        assert counts.max() > NT, "the skewed case should put several token tiles on one expert"
    # a second call (the masks and the counter are cleared per call) gives the same layer output
    y2 = layer.forward(to_dev_bf16(x, DEV), topk_idx=idx)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
