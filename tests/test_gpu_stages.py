"""Stage-by-stage parity of the CUDA library (through the C ABI) with the CPU oracle.

Integer and byte outputs (quantised codes and scales, top-k indices, the
permutation) must be bit-exact; floating-point outputs stay within the
tolerances stated per test.
"""
import numpy as np
import pytest
import torch

import lmoe_inputs as gen
import oracle
from _util import bf16_to_f64, canonical_to_tc, from_dev_bf16, pair_row_err, to_dev_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _special_weight_rows(K):
    """Blocks that hit rounding ties, saturation, zeros, tiny and negative values."""
    rows = []
    ties = np.array([4.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, 0.1, -0.1, 0.0, -0.0, 6.0,
                     7.0, 5.5, 0.2500001, 4.9999, 3.0, 2.0, 1.0, 0.5, -1.5, -3.5, -2.5, 1.4999, 0.7499, 0.2499, 3.25,
                     -6.5], np.float32)
    for scale in (1.0, 2.0 ** -60, 2.0 ** 40, 2.0 ** -120):
        r = np.zeros(K, np.float32)
        r[:32] = ties * np.float32(scale)
        rows.append(r)
    z = np.zeros(K, np.float32)
    z[32:64] = 1e-42  # subnormal block
    rows.append(z)
    return np.stack(rows)


@pytest.mark.parametrize("nmat,rows,K", [(1, 5, 256), (3, 200, 96), (2, 128, 3584), (4, 64, 512), (1, 512, 64)])
def test_quant_mxfp4_bit_exact(cuda_lib, nmat, rows, K):
    lmoe = cuda_lib
    rng = np.random.default_rng(nmat * 1000 + rows + K)
    w = (rng.standard_normal((nmat, rows, K)) * np.exp2(rng.integers(-30, 30, (nmat, rows, 1)))).astype(np.float32)
    sp = _special_weight_rows(K)
    n = min(rows, sp.shape[0])
    w[0, :n] = sp[:n]
    wd = torch.from_numpy(w).to(DEV)
    q, s = lmoe.quant_mxfp4(wd, lmoe.LAYOUT_CANONICAL)
    qt, st = lmoe.quant_mxfp4(wd, lmoe.LAYOUT_TC)
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_mxfp4(w.reshape(nmat * rows, K))
    np.testing.assert_array_equal(s.cpu().numpy(), os_.reshape(-1))
    np.testing.assert_array_equal(q.cpu().numpy(), oq.reshape(-1))
    rq, rs = canonical_to_tc(oq, os_, nmat, rows, K)
    np.testing.assert_array_equal(qt.cpu().numpy(), rq)
    np.testing.assert_array_equal(st.cpu().numpy(), rs)


@pytest.mark.parametrize("rows,K", [(1, 32), (7, 512), (64, 3584), (33, 96)])
def test_quant_mxfp8_bit_exact(cuda_lib, rows, K):
    lmoe = cuda_lib
    x = gen.normal_bf16(1, 40 + rows, 0, rows * K, 1.0).reshape(rows, K)
    if rows >= 4:
        x[0, :32] = 0
        mids = np.array([1.0625, 1.1875, 448.0, 460.0, 2 ** -9, 2 ** -10, 1.5 * 2 ** -9, -1.0625, 0.1, -0.1, 256.0,
                         300.0, 1e-3, -7.0, 3.0, 5.0], np.float32) / 256.0
        mids = np.concatenate([mids, np.float32([1.0 / 256.0 * 2.0])])  # amax 2/256 -> X = -15
        row = np.zeros(32, np.float32)
        row[:mids.size] = mids
        row[-1] = 1.0 / 256 * 1.75
        x[1, :32] = (row.view(np.uint32) >> 16).astype(np.uint16)
        x[2, :] = gen.normal_bf16(2, 9, 0, K, 1e-36)  # clamped scale byte, e4m3 subnormals
        x[3, :] = gen.normal_bf16(2, 10, 0, K, 1e30)
    q, s = lmoe.quant_mxfp8(to_dev_bf16(x, DEV))
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_mxfp8(x)
    np.testing.assert_array_equal(s.cpu().numpy(), os_)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)


def _route_case(lmoe, wl):
    x = gen.x_bf16(wl)
    Wr = gen.router_f32(wl)
    bias = gen.router_bias(wl)
    bd = None if bias is None else torch.from_numpy(bias).to(DEV)
    logits, idx, w = lmoe.route(to_dev_bf16(x, DEV), torch.from_numpy(Wr).to(DEV), wl.k, bias=bd)
    torch.cuda.synchronize()
    return x, Wr, bias, logits.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


WIDE = {  # more than 896 experts: 64 logits per lane in the selecting warp
    "wide_small_T": gen.custom("wide_small_T", T=40, d=512, I=64, E=1536),   # split-K + reduce/top-k
    "wide_large_T": gen.custom("wide_large_T", T=2048, d=512, I=64, E=1536),  # one-pass GEMM + top-k
}


@pytest.mark.parametrize("name", ["tiny", "decode", "skewed_small", "wide_small_T", "wide_large_T"])
def test_route_topk_exact_given_logits(cuda_lib, name):
    lmoe = cuda_lib
    wl = gen.WORKLOADS.get(name) or WIDE.get(name) or gen.custom(name, T=512, d=3584, I=512, zipf_s=1.2,
                                                                   zipf_beta=0.18)
    x, Wr, bias, lg, idx, w = _route_case(lmoe, wl)
    # the GPU's fp32 logits are close to the oracle's (fp32 accumulation order only)
    ref = oracle.router_logits(x, Wr, bias)
    assert np.max(np.abs(lg - ref)) <= 1e-4 * np.sqrt((ref.astype(np.float64) ** 2).mean())
    # given identical logits, indices are bit-exact and weights within 1e-6
    ridx, rw = oracle.topk_softmax(lg, wl.k)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=1e-6, atol=1e-9)
    # fully independent routing differs only on near-ties of the 16th/17th logit
    oidx, _ = oracle.topk_softmax(ref, wl.k)
    bad = np.flatnonzero((np.sort(oidx, 1) != np.sort(idx, 1)).any(1))
    for t in bad:
        s = np.sort(ref[t].astype(np.float64))[::-1]
        assert s[wl.k - 1] - s[wl.k] <= 1e-5 * np.sqrt((ref[t].astype(np.float64) ** 2).mean())


def test_topk_ties_and_signed_zero(cuda_lib):
    lmoe = cuda_lib
    rng = np.random.default_rng(11)
    T, E, k = 40, 896, 16
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[0] = 0.0
    l[1, ::2] = -0.0
    l[2] = np.round(l[2] * 2) / 2
    l[3, 100:140] = 7.0
    l[4] = -1e30
    l[5, 895] = 50.0
    # rows 6 and 7: exactly 64 and 65 values at or above the 16th largest of
    # the 32 lane maxima (lane j holds experts j, j+32, ...), the extra ones
    # tied at that bound: the selection's compacted-candidate limit and the
    # first count past it
    for r, extra in ((6, 48), (7, 49)):
        row = (np.float32(-10.0) - rng.random(E).astype(np.float32)).astype(np.float32)
        row[:32] = np.float32(1.0) + np.float32(0.01) * np.arange(32, dtype=np.float32)
        n, i = 0, 1
        while n < extra:
            for lane in range(17, 32):
                if n < extra:
                    row[lane + 32 * i] = row[16]
                    n += 1
            i += 1
        l[r] = row
    for E2, k2 in ((896, 16), (32, 32), (1, 1), (2048, 16), (300, 5)):
        ll = l[:, :E2] if E2 <= E else np.tile(l, (1, 3))[:, :E2].copy()
        idx, w = lmoe.topk_from_logits(torch.from_numpy(np.ascontiguousarray(ll)).to(DEV), k2)
        torch.cuda.synchronize()
        ridx, rw = oracle.topk_softmax(ll, k2)
        np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
        np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-6, atol=1e-9)


def _warp_bound_row(rng, E, extra):
    """A logits row whose 16th largest 32-expert group maximum is 1.0 (groups
    0..15 peak at 1.0 + 0.01 g, the rest lie below -10), with `extra` more
    values tied at 1.0 in the groups' other slots: 16 + extra values at or
    above the bound."""
    row = (np.float32(-10.0) - rng.random(E).astype(np.float32)).astype(np.float32)
    for g in range(16):
        row[32 * g] = np.float32(1.0) + np.float32(0.01) * np.float32(g)
    n = 0
    for g in range(1, 16):
        for j in range(1, 32):
            if n < extra:
                row[32 * g + j] = np.float32(1.0)
                n += 1
    assert n == extra
    return row


def test_split_k_route_topk_ties(cuda_lib):
    """The split-K router's reduction + top-k kernel (small batches) on
    crafted logits: token t's row of x is one-hot at column t, so its logits
    are exactly column t of the router weights.  Rows: all equal (every
    expert a candidate), signed zeros, many ties, exactly 64 and 65 values at
    the bound the block's candidate narrowing uses (16th largest maximum of the
    32-expert groups), group maxima tied at that bound, and a plain row."""
    lmoe = cuda_lib
    rng = np.random.default_rng(23)
    T, d, E, k = 8, 512, 896, 16
    cols = [np.zeros(E, np.float32)]
    r = rng.standard_normal(E).astype(np.float32)
    r[::2] = -0.0
    cols.append(r)
    cols.append((np.round(rng.standard_normal(E) * 2) / 2).astype(np.float32))
    cols.append(_warp_bound_row(rng, E, 48))
    cols.append(_warp_bound_row(rng, E, 49))
    r = (np.float32(-10.0) - rng.random(E).astype(np.float32)).astype(np.float32)
    r[32 * np.arange(20)] = np.float32(2.0)  # 20 group maxima tied, the bound among them
    cols.append(r)
    r = rng.standard_normal(E).astype(np.float32)
    r[100:140] = 7.0
    cols.append(r)
    cols.append(rng.standard_normal(E).astype(np.float32))
    Wr = (rng.standard_normal((E, d)) * 0.05).astype(np.float32)
    for t, c in enumerate(cols):
        Wr[:, t] = c
    x = np.zeros((T, d), np.uint16)
    x[np.arange(T), np.arange(T)] = 0x3F80  # bf16 1.0
    logits, idx, w = lmoe.route(to_dev_bf16(x, DEV), torch.from_numpy(Wr).to(DEV), k)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    # the logits are the crafted columns (signed zeros may come back as +0)
    np.testing.assert_array_equal(lg, Wr[:, :T].T + np.float32(0.0))
    ridx, rw = oracle.topk_softmax(lg, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("T,E,k,skew", [(8, 896, 16, 0), (64, 896, 16, 0), (300, 896, 16, 1), (8192, 896, 16, 1),
                                        (1000, 2048, 8, 0), (1, 4, 4, 0), (0, 896, 16, 0), (5000, 7, 3, 0)])
def test_permute_bit_exact(cuda_lib, T, E, k, skew):
    lmoe = cuda_lib
    rng = np.random.default_rng(T + E + k)
    if T:
        score = rng.standard_normal((T, E)) + (skew * 3.0 * -np.log1p(np.arange(E)))[None, :]
        idx = np.argsort(-score, 1, kind="stable")[:, :k].astype(np.int32)
    else:
        idx = np.zeros((0, k), np.int32)
    counts, offsets, perm, inv, ws = lmoe.permute(torch.from_numpy(idx).to(DEV), E)
    torch.cuda.synchronize()
    assert lmoe.last_device_status(ws) == 0
    rc, ro, rp, ri = oracle.permute(idx, E)
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(perm.cpu().numpy(), rp)
    np.testing.assert_array_equal(inv.cpu().numpy(), ri)


def test_permute_flags_out_of_range_ids(cuda_lib):
    lmoe = cuda_lib
    idx = np.tile(np.arange(16, dtype=np.int32), (10, 1))
    idx[3, 5] = 896  # out of range
    counts, offsets, perm, inv, ws = lmoe.permute(torch.from_numpy(idx).to(DEV), 896)
    torch.cuda.synchronize()
    assert lmoe.last_device_status(ws) == lmoe.ERR_DEVICE_CHECK
    assert int(inv[3 * 16 + 5]) == -1 and int(offsets[-1]) == 159


def test_prepare_router_planes_sum_to_fp32(cuda_lib):
    """lmoe_prepare_router: hi = bf16_rne(W), then the two residual planes; the
    three bf16 planes add up to the fp32 weights exactly (24 significand
    bits), across a wide exponent range."""
    lmoe = cuda_lib
    rng = np.random.default_rng(5)
    E, d = 40, 192
    W = (rng.standard_normal((E, d)) * np.exp2(rng.integers(-60, 60, (E, d)))).astype(np.float32)
    W3 = lmoe.prepare_router(torch.from_numpy(W).to(DEV))
    torch.cuda.synchronize()
    planes = bf16_to_f64(from_dev_bf16(W3)).reshape(3, E, d)
    np.testing.assert_array_equal(planes.sum(0), W.astype(np.float64))
    hi = torch.from_numpy(W).to(torch.bfloat16).float().numpy().astype(np.float64)  # RNE
    np.testing.assert_array_equal(planes[0], hi)


def test_combine_slot_order_fp32(cuda_lib):
    lmoe = cuda_lib
    rng = np.random.default_rng(12)
    for T, d, k in ((5, 512, 16), (64, 3584, 16), (3, 128, 1), (1, 256, 32)):
        P = T * k
        yp = (rng.standard_normal((P, d)) * 10).astype(np.float32)
        inv = rng.permutation(P).astype(np.int32)
        y = lmoe.combine(torch.from_numpy(yp).to(DEV), torch.from_numpy(inv).to(DEV), T, k)
        torch.cuda.synchronize()
        acc = np.zeros((T, d), np.float32)
        for j in range(k):
            acc = acc + yp[inv.reshape(T, k)[:, j]]
        ref = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(from_dev_bf16(y), ref)


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_expert_ffn_against_oracle_per_pair(cuda_lib, name):
    from _util import device_bank
    lmoe = cuda_lib
    wl = gen.WORKLOADS["tiny"] if name == "tiny" else gen.custom("ragged", T=37, d=256, I=96, E=40, k=6)
    x = gen.x_bf16(wl)
    xd = to_dev_bf16(x, DEV)
    logits, idx, w = lmoe.route(xd, torch.from_numpy(gen.router_f32(wl)).to(DEV), wl.k)
    counts, offsets, perm, inv, _ = lmoe.permute(idx, wl.E)
    xq, xs = lmoe.quant_mxfp8(xd)
    bank = device_bank(wl, DEV)
    yp, _ = lmoe.expert_ffn(xq, xs, bank, offsets, perm, w, wl.k)
    torch.cuda.synchronize()
    yp, perm_h, idx_h, w_h = yp.cpu().numpy(), perm.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()
    ob = oracle.quantize_experts(wl, experts=np.unique(idx_h))
    worst = 0.0
    for q in range(0, wl.P, max(1, wl.P // 64)):
        p = perm_h[q]
        t, j = divmod(int(p), wl.k)
        e = int(idx_h[t, j])
        ref = float(w_h[t, j]) * oracle.expert_ffn_token(x[t], ob, e, wl.d, wl.I)
        worst = max(worst, pair_row_err(yp[q], ref, x[t], e, float(w_h[t, j]), ob, wl.d, wl.I, 1e-2))
    assert np.isfinite(worst)


def _ffn_case(lmoe, wl, idx, seed=0):
    """Expert FFN stage on a given routing; checks sampled pairs against the oracle."""
    from _util import device_bank
    rng = np.random.default_rng(seed)
    x = gen.x_bf16(wl)
    xd = to_dev_bf16(x, DEV)
    w = rng.uniform(0.01, 1.0, idx.shape).astype(np.float32)
    counts, offsets, perm, inv, _ = lmoe.permute(torch.from_numpy(idx).to(DEV), wl.E)
    xq, xs = lmoe.quant_mxfp8(xd)
    bank = device_bank(wl, DEV)
    yp, ws = lmoe.expert_ffn(xq, xs, bank, offsets, perm, torch.from_numpy(w).to(DEV), wl.k)
    torch.cuda.synchronize()
    assert lmoe.last_device_status(ws) == 0
    yp, perm_h = yp.cpu().numpy(), perm.cpu().numpy()
    ob = oracle.quantize_experts(wl, experts=np.unique(idx))
    worst = 0.0
    qs = sorted(set(list(range(0, wl.P, max(1, wl.P // 48))) + [wl.P - 1]))
    for q in qs:
        t, j = divmod(int(perm_h[q]), wl.k)
        e = int(idx[t, j])
        ref = float(w[t, j]) * oracle.expert_ffn_token(x[t], ob, e, wl.d, wl.I)
        worst = max(worst, pair_row_err(yp[q], ref, x[t], e, float(w[t, j]), ob, wl.d, wl.I, 1e-2))
    return worst


def test_expert_ffn_multi_tile_and_last_expert_small_tiles(cuda_lib):
    """Token tiles of 32 (few tokens per expert): an expert with 75 tokens spans
    three tiles; the last expert's weight rows run past the bank (I = 64)."""
    wl = gen.custom("multi32", T=80, d=256, I=64, E=60, k=4)
    idx = np.zeros((wl.T, wl.k), np.int32)
    for t in range(wl.T):
        idx[t] = [59, (t % 50) + 1, (t % 7) + 51, 0 if t < 75 else 58]
    assert lmoe_nt(cuda_lib, wl) == 32
    _ffn_case(cuda_lib, wl, idx)


def test_expert_ffn_large_tiles_ragged_I(cuda_lib):
    """Token tiles of 96 (many tokens per expert), experts with 1..~300
    tokens, I = 160 (a partial 128-row tile and a partial K chunk in the down
    GEMM)."""
    wl = gen.custom("multi96", T=600, d=384, I=160, E=8, k=2)
    rng = np.random.default_rng(3)
    idx = np.zeros((wl.T, wl.k), np.int32)
    for t in range(wl.T):
        idx[t] = rng.choice(7, 2, replace=False, p=np.array([50, 20, 10, 10, 5, 4, 1.0]) / 100) + (t == 0)
    idx[0] = [7, 0]  # expert 7: a single token
    assert lmoe_nt(cuda_lib, wl) == 96
    _ffn_case(cuda_lib, wl, idx)


def lmoe_nt(lmoe, wl):
    # the token tile the library picks by the mean pairs per expert
    P, E = wl.P, wl.E
    return 16 if P <= 4 * E else 32 if P <= 16 * E else 96
