"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against the format definitions, closed
forms, a brute-force or library computation written here in numpy, or
invariants that any correct result must satisfy.  None of them needs a GPU.
"""
import math
import os
import struct

import numpy as np
import pytest

import lmoe_inputs as gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- independent numpy restatements of the formats ---------------------------------

def e2m1_closed_form(code):
    s = -1.0 if code & 8 else 1.0
    e, m = (code >> 1) & 3, code & 1
    return s * (m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2))


def e4m3_closed_form(code):
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * m / 8 * 2.0 ** -6
    return s * (1 + m / 8) * 2.0 ** (e - 7)


E2M1_MAG = np.array([e2m1_closed_form(c) for c in range(8)])
E4M3_MAG = np.array([e4m3_closed_form(c) for c in range(127)])


def np_nearest_even(a, grid):
    """Brute force: distance to every grid point; ties -> even index; saturate."""
    a = np.asarray(a, np.float64)
    dist = np.abs(a[..., None] - grid)
    best = dist.min(-1, keepdims=True)
    cand = dist == best
    # among equal-distance candidates prefer an even index
    even = cand & (np.arange(grid.size) % 2 == 0)
    idx = np.where(even.any(-1), np.argmax(even, -1), np.argmax(cand, -1))
    return np.where(a >= grid[-1], grid.size - 1, idx)


def floor_log2_f32(v):
    """floor(log2 v) of a positive fp32 value from its bit pattern."""
    bits = struct.unpack("<I", struct.pack("<f", v))[0]
    ex = (bits >> 23) & 0xFF
    man = bits & 0x7FFFFF
    if ex == 0:
        return man.bit_length() - 1 - 149
    return ex - 127


def np_scale_bytes(amax, emax):
    out = []
    for a in np.asarray(amax, np.float32).ravel():
        if a == 0:
            out.append(0)
        else:
            out.append(int(min(254, max(0, floor_log2_f32(float(a)) - emax + 127))))
    return np.array(out, np.uint8).reshape(np.shape(amax))


def np_quant(x, emax, grid, signbit_shift):
    """MX block quantisation of float rows along the last axis, block 32."""
    x = np.asarray(x, np.float64)
    rows, K = x.shape
    blk = x.reshape(rows, K // 32, 32)
    amax = np.abs(blk).max(-1).astype(np.float32)  # exact: values are fp32 or bf16
    sb = np_scale_bytes(amax, emax)
    v = blk / np.exp2(sb.astype(np.float64) - 127)[..., None]
    mag = np_nearest_even(np.abs(v), grid)
    code = mag | (np.signbit(v).astype(np.int64) << signbit_shift)
    return code.reshape(rows, K).astype(np.uint8), sb


def bf16_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---- codecs ---------------------------------------------------------------------

def test_e2m1_decode_matches_typed_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_grid.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 16
    for code, val in rows:
        got = oracle.e2m1_value(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e4m3_decode_all_codes_closed_form():
    for c in range(256):
        ref, got = e4m3_closed_form(c), oracle.e4m3_value(c)
        if math.isnan(ref):
            assert math.isnan(got) and c in (0x7F, 0xFF)
        else:
            assert got == ref, hex(c)
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9 and oracle.e4m3_value(0x08) == 2.0 ** -6


def test_e8m0_decode():
    for s in range(255):
        assert oracle.e8m0_value(s) == 2.0 ** (s - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_encoders_round_trip_every_code():
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_value(c)) == c
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c


def test_rounding_ties_and_saturation_typed_cases():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "rounding_ties.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) > 20
    for fmt, val, code in rows:
        enc = oracle.e2m1_encode if fmt == "e2m1" else oracle.e4m3_encode
        assert enc(float(val)) == int(code), (fmt, val)


def test_encoders_match_brute_force_nearest():
    rng = np.random.default_rng(1)
    a = np.concatenate([rng.uniform(0, 7, 4000), rng.uniform(0, 1, 2000),
                        (np.arange(15) + 0.5) / 2])  # includes all e2m1 midpoints
    ref = np_nearest_even(a, E2M1_MAG)
    got = np.array([oracle.e2m1_encode(float(v)) for v in a])
    np.testing.assert_array_equal(got, ref)
    b = np.concatenate([np.exp2(rng.uniform(-12, 9.5, 6000)), (E4M3_MAG[1:] + E4M3_MAG[:-1]) / 2])
    ref = np_nearest_even(b, E4M3_MAG)
    got = np.array([oracle.e4m3_encode(float(v)) for v in b])
    np.testing.assert_array_equal(got, ref)


def test_scale_byte_against_bit_pattern_exponent():
    rng = np.random.default_rng(2)
    vals = np.concatenate([np.exp2(rng.uniform(-149, 127, 3000)).astype(np.float32),
                           np.float32([1.0, 2.0, 3.999, 4.0, 6.0, 448.0, 2.0 ** -126, 2.0 ** -149, 1e-40])])
    vals = vals[vals > 0]
    for emax in (2, 8):
        ref = np_scale_bytes(vals, emax)
        got = np.array([oracle.scale_byte(float(v), emax) for v in vals], np.uint8)
        np.testing.assert_array_equal(got, ref)
    assert oracle.scale_byte(0.0, 2) == 0 and oracle.scale_byte(0.0, 8) == 0
    # amax 1.0 -> X = -2 (e2m1) -> byte 125; amax 6 -> floor(log2 6)=2 -> byte 127
    assert oracle.scale_byte(1.0, 2) == 125 and oracle.scale_byte(6.0, 2) == 127


# ---- block quantisation ----------------------------------------------------------

def test_quant_mxfp4_matches_numpy_restatement():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((24, 256)) * np.exp2(rng.integers(-20, 20, (24, 1)))).astype(np.float32)
    w[0, :32] = 0.0                        # all-zero block
    w[1, :32] = 0.0
    w[1, 0] = 7.0                          # saturates to 6
    w[2, 32:64] = 1e-42                    # subnormal block
    q, s = oracle.quant_mxfp4(w)
    ref_code, ref_s = np_quant(w, 2, E2M1_MAG, 3)
    np.testing.assert_array_equal(s, ref_s)
    lo, hi = q & 15, q >> 4
    np.testing.assert_array_equal(lo, ref_code[:, 0::2])   # element 2i in the low nibble
    np.testing.assert_array_equal(hi, ref_code[:, 1::2])
    dq = oracle.dequant_mxfp4(q, s)
    assert dq[1, 0] == 6.0 and s[0, 0] == 0 and np.all(dq[0, :32] == 0)


def test_quant_mxfp4_round_trip_exact_every_code_and_scale():
    # blocks whose largest magnitude is 4 or 6 (so the recomputed scale is the
    # same), each block at scale byte sb, every code present
    codes = np.tile(np.arange(16), 2)
    for sb in range(0, 253):
        for top in (6, 7):  # top code 6 -> 4.0, 7 -> 6.0
            blk = codes.copy()
            blk[0] = top
            blk[1:][(blk[1:] & 7) > top] = 0
            vals = np.array([e2m1_closed_form(int(c)) for c in blk]) * 2.0 ** (sb - 127)
            w = vals.astype(np.float32)
            assert np.all(w.astype(np.float64) == vals)       # exactly representable
            q, s = oracle.quant_mxfp4(w[None, :])
            assert s[0, 0] == sb
            assert np.array_equal(oracle.dequant_mxfp4(q, s)[0], vals)


def test_quant_mxfp8_matches_numpy_restatement():
    rng = np.random.default_rng(4)
    x = gen.normal_bf16(0, 77, 0, 16 * 512, 1.0).reshape(16, 512)
    x[0, :32] = 0                                     # zero block
    x[1, :32] = np.array([0x3F80], np.uint16)         # all 1.0
    x[2, :] = gen.normal_bf16(0, 78, 0, 512, 1e-30)   # tiny values: clamped scale
    q, s = oracle.quant_mxfp8(x)
    ref_code, ref_s = np_quant(bf16_to_f64(x), 8, E4M3_MAG, 7)
    np.testing.assert_array_equal(s, ref_s)
    np.testing.assert_array_equal(q, ref_code)
    assert s[1, 0] == 127 - 8 and q[1, 0] == 0x78  # 1.0 / 2^-8 = 256 = e4m3 0x78
    del rng


def test_mxfp8_round_trip_exact_every_code_and_scale():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    for sb in range(0, 247, 3):
        for top in (0x78, 0x7E):  # 256 and 448 are the largest magnitudes of the block
            blk = np.resize(codes[(codes & 0x7F) <= top], 32)
            blk[0] = top
            vals = np.array([e4m3_closed_form(int(c)) for c in blk]) * 2.0 ** (sb - 127)
            q, s = oracle.quant_mxfp8_f64(vals[None, :])
            assert s[0, 0] == sb
            assert np.array_equal(oracle.dequant_mxfp8(q, s)[0], vals)


# ---- routing -----------------------------------------------------------------------

def test_router_logits_match_numpy_matmul():
    wl = gen.custom("t", T=5, d=256, I=64, E=40)
    x = gen.x_bf16(wl)
    Wr = gen.router_f32(wl)
    bias = np.linspace(-1, 1, 40).astype(np.float32)
    ref = (bf16_to_f64(x) @ Wr.astype(np.float64).T).astype(np.float32)
    got = oracle.router_logits(x, Wr)
    np.testing.assert_array_max_ulp(got, ref, maxulp=1)
    got_b = oracle.router_logits(x, Wr, bias)
    np.testing.assert_array_max_ulp(got_b, (got + bias).astype(np.float32), maxulp=0)


def test_topk_matches_full_sort_with_ties_and_signed_zero():
    rng = np.random.default_rng(5)
    T, E, k = 64, 896, 16
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[0, :] = 0.0                                  # all equal: ids 0..15
    l[1, ::2] = -0.0                               # +0 / -0 compare equal
    l[1, 1::2] = 0.0
    l[2] = np.round(l[2] * 2) / 2                  # many exact ties
    l[3, 100:130] = 5.0
    idx, w = oracle.topk_softmax(l, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -l[t].astype(np.float64)))
        np.testing.assert_array_equal(idx[t], order[:k])
    np.testing.assert_array_equal(idx[0], np.arange(16))
    np.testing.assert_array_equal(idx[1], np.arange(16))
    np.testing.assert_array_equal(idx[3], np.arange(100, 116))


def test_softmax_identities():
    rng = np.random.default_rng(6)
    l = (rng.standard_normal((32, 896)) * 3).astype(np.float32)
    idx, w = oracle.topk_softmax(l, 16)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1) < 1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)
    sel = np.take_along_axis(l, idx, 1).astype(np.float64)
    for i in range(16):
        np.testing.assert_allclose(w[:, i] / w[:, 0], np.exp(sel[:, i] - sel[:, 0]), rtol=2e-6)
    idx1, w1 = oracle.topk_softmax(l, 1)
    assert np.all(w1 == 1.0)


def test_permute_is_stable_counting_sort():
    rng = np.random.default_rng(7)
    T, k, E = 300, 16, 896
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle.topk_softmax(logits, k)
    counts, offsets, perm, inv = oracle.permute(idx, E)
    flat = idx.ravel()
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k
    np.testing.assert_array_equal(np.diff(offsets), counts)
    np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(inv[perm], np.arange(T * k))
    for e in np.flatnonzero(counts)[:50]:
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


# ---- experts ---------------------------------------------------------------------

def _tiny_bank(wl, experts):
    return oracle.quantize_experts(wl, experts=experts)


def np_swiglu_layer(x_bf16, idx, w, bank, wl, tokens):
    """numpy restatement: decode weights from the typed grid, MXFP8 via np_quant."""
    d, I = wl.d, wl.I
    gq, gs, uq, us, dq, ds = bank.arrays

    def deq4(q, s):
        codes = np.stack([q & 15, q >> 4], -1).reshape(*q.shape[:-1], -1)
        vals = np.array([e2m1_closed_form(c) for c in range(16)])[codes]
        return vals * np.repeat(np.exp2(s.astype(np.float64) - 127), 32, -1)

    def mx8(v):
        c, s = np_quant(v[None, :], 8, E4M3_MAG, 7)
        mag = np.array([e4m3_closed_form(int(cc) & 0x7F) for cc in c[0]])
        sign = np.where(c[0] & 0x80, -1.0, 1.0)
        return sign * mag * np.repeat(np.exp2(s[0].astype(np.float64) - 127), 32)

    out = []
    for t in tokens:
        xh = mx8(bf16_to_f64(x_bf16[t]))
        y = np.zeros(d)
        for j in range(idx.shape[1]):
            e = idx[t, j]
            g = deq4(gq[e], gs[e]) @ xh
            u = deq4(uq[e], us[e]) @ xh
            h = g / (1 + np.exp(-g)) * u
            y += float(w[t, j]) * (deq4(dq[e], ds[e]) @ mx8(h))
        out.append(y)
    return np.array(out)


def test_moe_sparse_equals_dense_brute_force_tiny():
    wl = gen.WORKLOADS["tiny"]
    x = gen.x_bf16(wl)
    logits = oracle.router_logits(x, gen.router_f32(wl))
    idx, w = oracle.topk_softmax(logits, wl.k)
    bank = oracle.quantize_experts(wl)  # all 896 experts (dense evaluates every one)
    toks = np.array([0, 3, 7], np.int32)
    _, ys = oracle.moe_tokens(x, idx, w, bank, wl.d, wl.E, wl.I, tokens=toks, want_f64=True)
    yd = oracle.moe_dense(x, idx, w, bank, wl.d, wl.E, wl.I, tokens=toks)
    scale = np.sqrt((yd ** 2).mean(1, keepdims=True))
    assert np.max(np.abs(ys - yd) / scale) < 1e-12


def test_moe_matches_numpy_restatement():
    wl = gen.custom("small", T=4, d=128, I=64, E=12, k=3)
    x = gen.x_bf16(wl)
    logits = oracle.router_logits(x, gen.router_f32(wl))
    idx, w = oracle.topk_softmax(logits, wl.k)
    bank = oracle.quantize_experts(wl)
    y16, yf = oracle.moe_tokens(x, idx, w, bank, wl.d, wl.E, wl.I, want_f64=True)
    ref = np_swiglu_layer(x, idx, w, bank, wl, range(wl.T))
    scale = np.sqrt((ref ** 2).mean(1, keepdims=True))
    assert np.max(np.abs(yf - ref) / scale) < 1e-12
    np.testing.assert_array_equal(y16, oracle.round_bf16(yf))


def test_single_expert_reduces_to_dense_swiglu_ffn():
    """k = E = 1 with w = 1: a plain SwiGLU FFN on the decoded weights."""
    wl = gen.custom("one", T=3, d=64, I=32, E=1, k=1)
    x = gen.x_bf16(wl)
    idx = np.zeros((3, 1), np.int32)
    w = np.ones((3, 1), np.float32)
    bank = oracle.quantize_experts(wl)
    _, yf = oracle.moe_tokens(x, idx, w, bank, wl.d, wl.E, wl.I, want_f64=True)
    for t in range(3):
        np.testing.assert_allclose(yf[t], oracle.expert_ffn_token(x[t], bank, 0, wl.d, wl.I), rtol=0, atol=0)
    ref = np_swiglu_layer(x, idx, w, bank, wl, range(3))
    np.testing.assert_allclose(yf, ref, rtol=1e-12, atol=1e-14)
    x0 = np.zeros_like(x)
    _, y0 = oracle.moe_tokens(x0, idx, w, bank, wl.d, wl.E, wl.I, want_f64=True)
    assert np.all(y0 == 0)


def test_linear_bf16_matches_numpy():
    rng = np.random.default_rng(8)
    x = gen.normal_bf16(0, 90, 0, 6 * 96, 1.0).reshape(6, 96)
    W = gen.normal_bf16(0, 91, 0, 40 * 96, 0.1).reshape(40, 96)
    ref = oracle.round_bf16(bf16_to_f64(x) @ bf16_to_f64(W).T)
    np.testing.assert_array_equal(oracle.linear_bf16(x, W), ref)
    del rng


# ---- bf16 rounding of the layer output and the projections ------------------------

def test_round_bf16_typed_cases():
    """Ties, carries, overflow, subnormals and signed zeros worked out from
    the bf16 format definition (tests/golden/bf16_rounding.txt), including
    doubles just off a midpoint that an fp32 pass would turn into a tie."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "bf16_rounding.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) >= 30
    v = np.array([float.fromhex(r[0]) for r in rows])
    want = np.array([int(r[1], 16) for r in rows], np.uint16)
    got = oracle.round_bf16(v)
    bad = [(rows[i][0], rows[i][1], f"{got[i]:04x}") for i in np.nonzero(got != want)[0]]
    assert not bad, bad


def test_round_bf16_matches_torch_on_every_kind_of_fp32_input():
    """On inputs that are fp32 values, rounding the double once equals
    torch's fp32 -> bf16 conversion (round to nearest even; no double
    rounding is possible): random bit patterns over the whole finite range,
    every bf16 midpoint and its fp32 neighbours, fp32 subnormals, +-0."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2024)
    pats = [rng.integers(0, 2 ** 32, size=3_000_000, dtype=np.uint64).astype(np.uint32)]
    b = np.arange(0, 0x10000, dtype=np.uint32)
    mid = (b << 16) | 0x8000
    pats += [mid, mid - 1, mid + 1]
    pats.append(rng.integers(0, 0x800000, size=200_000, dtype=np.uint64).astype(np.uint32))  # subnormals
    pats.append(np.array([0, 0x80000000, 1, 0x80000001, 0x7F7F7FFF, 0x7F7F8000, 0xFF7F8000], np.uint32))
    u = np.concatenate(pats)
    u = u[(u & 0x7F800000) != 0x7F800000]  # finite inputs only
    f = u.view(np.float32)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(f.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(f"{u[i]:08x}", f"{got[i]:04x}", f"{want[i]:04x}") for i in bad[:10]]


def test_round_bf16_of_doubles_is_not_rounded_through_fp32():
    """Doubles strictly between a bf16 midpoint and its fp32 neighbours round
    to the bf16 value on their own side of the midpoint; a rounding that went
    through fp32 first would land on the tie and pick the even side for
    half of them."""
    rng = np.random.default_rng(7)
    b = rng.integers(0x0080, 0x7F7F, size=20_000).astype(np.uint32)  # positive normal bf16, not the largest
    lo = ((b << 16)).view(np.float32).astype(np.float64)
    hi = (((b + 1) << 16)).view(np.float32).astype(np.float64)
    mid = (lo + hi) / 2
    tiny = (hi - lo) * 2.0 ** -30  # far below an fp32 ulp there
    up = oracle.round_bf16(mid + tiny)
    down = oracle.round_bf16(mid - tiny)
    np.testing.assert_array_equal(up, (b + 1).astype(np.uint16))
    np.testing.assert_array_equal(down, b.astype(np.uint16))
    np.testing.assert_array_equal(oracle.round_bf16(-(mid + tiny)), ((b + 1) | 0x8000).astype(np.uint16))


# ---- the full-FP4 activation mode (x and h rounded to MXFP4) ----------------------

def np_quant_f64(x, emax, grid, signbit_shift):
    """MX block quantisation of float64 rows: the scale exponent is
    floor(log2 amax) taken exactly from frexp of the double amax."""
    x = np.asarray(x, np.float64)
    rows, K = x.shape
    blk = x.reshape(rows, K // 32, 32)
    amax = np.abs(blk).max(-1)
    _, ex = np.frexp(amax)  # amax = m 2^ex, m in [0.5, 1)
    sb = np.where(amax == 0, 0, np.clip(ex - 1 - emax + 127, 0, 254)).astype(np.int64)
    v = blk / np.exp2(sb.astype(np.float64) - 127)[..., None]
    mag = np_nearest_even(np.abs(v), grid)
    code = mag | (np.signbit(v).astype(np.int64) << signbit_shift)
    return code.reshape(rows, K), sb.astype(np.uint8)


def test_quant_mxfp4_f64_matches_numpy_restatement():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((24, 256)) * np.exp2(rng.integers(-20, 20, size=(24, 1)))
    x[0, :32] = 0.0                                        # all-zero block
    x[1, :32] = 4.0 * (1 + 2.0 ** -40)                     # amax just above a power of two (not an fp32 value)
    x[2, :32] = 4.0 * (1 - 2.0 ** -40)                     # just below
    x[3, :32] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4)  # e2m1 ties at scale 1 (amax 6)
    x[4, 32:64] = -x[3, :32]
    codes, sb = np_quant_f64(x, 2, E2M1_MAG, 3)
    q, s = oracle.quant_mxfp4_f64(x)
    np.testing.assert_array_equal(s, sb)
    got = np.stack([q & 15, q >> 4], -1).reshape(24, 256)
    np.testing.assert_array_equal(got, codes)


def test_fp4_activation_mode_matches_numpy_restatement():
    wl = gen.custom("small_fp4", T=4, d=128, I=64, E=12, k=3)
    x = gen.x_bf16(wl)
    idx, w = oracle.topk_softmax(oracle.router_logits(x, gen.router_f32(wl)), wl.k)
    bank = oracle.quantize_experts(wl)
    y16, yf = oracle.moe_tokens(x, idx, w, bank, wl.d, wl.E, wl.I, want_f64=True, act=oracle.ACT_MXFP4)
    gq, gs, uq, us, dq, ds = bank.arrays

    def deq4(q, s):
        codes = np.stack([q & 15, q >> 4], -1).reshape(*q.shape[:-1], -1)
        vals = np.array([e2m1_closed_form(c) for c in range(16)])[codes]
        return vals * np.repeat(np.exp2(s.astype(np.float64) - 127), 32, -1)

    def mx4(v):
        c, s = np_quant_f64(v[None, :], 2, E2M1_MAG, 3)
        vals = np.array([e2m1_closed_form(int(cc)) for cc in c[0]])
        return vals * np.repeat(np.exp2(s[0].astype(np.float64) - 127), 32)

    for t in range(wl.T):
        xh = mx4(bf16_to_f64(x[t]))
        y = np.zeros(wl.d)
        for j in range(wl.k):
            e = idx[t, j]
            g = deq4(gq[e], gs[e]) @ xh
            u = deq4(uq[e], us[e]) @ xh
            y += float(w[t, j]) * (deq4(dq[e], ds[e]) @ mx4(g / (1 + np.exp(-g)) * u))
        np.testing.assert_allclose(yf[t], y, rtol=1e-12, atol=1e-12 * np.abs(y).max())
    np.testing.assert_array_equal(y16, oracle.round_bf16(yf))


def test_fp4_activation_mode_tolerance_study():
    """How far the full-FP4 variant's output lies from the MXFP8 layer's, on
    decode-shaped tokens (d = 3584, I = 512): several per cent of the row
    RMS, i.e. a different numerics regime than the MXFP8 layer's 1e-2 bar;
    GPU parity of the FP4 variant is therefore checked against this mode of
    the oracle, not against the MXFP8 layer."""
    wl = gen.custom("fp4_study", T=3, d=3584, I=512)
    x = gen.x_bf16(wl)
    idx, w = oracle.topk_softmax(oracle.router_logits(x, gen.router_f32(wl)), wl.k)
    bank = oracle.quantize_experts(wl, experts=np.unique(idx))
    _, y8 = oracle.moe_tokens(x, idx, w, bank, wl.d, wl.E, wl.I, want_f64=True)
    _, y4 = oracle.moe_tokens(x, idx, w, bank, wl.d, wl.E, wl.I, want_f64=True, act=oracle.ACT_MXFP4)
    rms = np.sqrt((y8 ** 2).mean(1))
    rel_rms = np.sqrt(((y4 - y8) ** 2).mean(1)) / rms
    rel_max = np.abs(y4 - y8).max(1) / rms
    print(f"FP4 vs MXFP8 activations: relative RMS difference {rel_rms.round(4)}, max {rel_max.round(3)}")
    assert np.all(rel_rms > 1e-2) and np.all(rel_rms < 0.3)
