"""Pins of the CPU oracle to facts outside itself.

Each test checks the oracle against something the pages or mathematics fix:
the magnitudes the TPU page prints, its piecewise-linear decode identity, the
OCP e2m1 bit definition, exact rational arithmetic, textbook routines (stable
argsort, dense matmul, logistic function, einsum) and closed forms.  No test
re-types the oracle's own formula.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from fp4_weight_grouped_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _golden_magnitudes(golden_dir):
    with open(os.path.join(golden_dir, "e2m1_magnitudes.txt")) as f:
        rows = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    return [Fraction(tok) for tok in rows[0].split()]


# ---------------------------------------------------------------- e2m1 decode

def test_e2m1_magnitudes_match_page(golden_dir):
    mags = _golden_magnitudes(golden_dir)
    assert len(mags) == 8
    for c in range(8):
        assert Fraction(oracle.e2m1_value(c)) == mags[c]
        assert Fraction(oracle.e2m1_value(c + 8)) == -mags[c]


def test_minus_zero_code_decodes_to_plus_zero():
    v = oracle.e2m1_value(8)
    assert v == 0.0 and math.copysign(1.0, v) == 1.0


def test_e2m1_piecewise_linear_identity_all_codes():
    # The TPU page's decode of the re-encoded integer q = +/-(2e+m):
    # v = 2q - clip(q, -6, 6) - 0.5 * clip(q, -4, 4).
    for c in range(16):
        q = (-1 if c & 8 else 1) * (c & 7)
        v = 2 * q - np.clip(q, -6, 6) - 0.5 * np.clip(q, -4, 4)
        assert oracle.e2m1_value(c) == v
        assert math.copysign(1.0, oracle.e2m1_value(c)) == math.copysign(1.0, v + 0.0)


def test_e2m1_matches_ocp_bit_definition():
    # OCP MX e2m1: exponent bias 1, one mantissa bit, subnormal when e == 0.
    for c in range(16):
        s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
        mag = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
        assert Fraction(oracle.e2m1_value(c)) == (-mag if s else mag)


# ------------------------------------------------------------------- bfloat16

def _bf16_rne_fraction(x: Fraction) -> Fraction:
    """Round to the bfloat16 grid by exhaustive rational arithmetic."""
    if x == 0:
        return Fraction(0)
    sgn = -1 if x < 0 else 1
    a = abs(x)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    q = max(e - 7, -133)              # 8 significant bits; fixed quantum below 2^-126
    scaled = abs(x) / Fraction(2) ** q
    fl = scaled.numerator // scaled.denominator
    rem = scaled - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sgn * fl * Fraction(2) ** q


def test_bf16_rounding_matches_rational_brute_force():
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 38, 2000))
    vals += [1 + 2 ** -8, 1 + 3 * 2 ** -8,                 # ties -> even
             math.ldexp(1.0, -133), math.ldexp(1.0, -134), math.ldexp(3.0, -135),
             math.ldexp(1.5, -127), 1e-45, -2.5e-39, 3.3e38, -3.4e38]
    for v in vals:
        bits = oracle.double_to_bf16(v)
        want = _bf16_rne_fraction(Fraction(v))
        if abs(want) >= Fraction(2) ** 128:
            assert bits & 0x7FFF == 0x7F80
        else:
            assert Fraction(oracle.bf16_to_double(bits)) == want, (v, hex(bits))


def test_bf16_rounding_agrees_with_float32_path():
    # For float32 inputs, rounding to bf16 is a plain bit operation; the
    # input generator implements it independently.
    rng = np.random.default_rng(2)
    x = rng.standard_normal(5000).astype(np.float32)
    ref = inputs.f32_to_bf16_bits(x)
    got = np.array([oracle.double_to_bf16(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_scaled_e2m1_is_exact_in_bf16_for_every_e8m0_exponent():
    # One expert, N=16 codes x K=256 columns: every code against scale bytes
    # 0..252 (exponents -127..125); the decoded bf16 must equal the exact value.
    codes_row = np.array([(c | (c << 4)) for c in range(16)] * 8, dtype=np.uint8)  # K/2 = 128
    s_bytes = np.arange(0, 253)
    for start in range(0, len(s_bytes), 8):
        chunk = s_bytes[start:start + 8]
        scales = np.full((1, 1, 8), chunk[-1], np.uint8)
        scales[0, 0, :len(chunk)] = chunk
        codes = codes_row.reshape(1, 1, 128)
        dec = oracle.decode_expert_bf16(codes, scales, 0)
        for k in range(256):
            c = k // 2 % 16
            s = int(scales[0, 0, k // 32])
            want = Fraction(oracle.e2m1_value(c)) * Fraction(2) ** (s - 127)
            assert Fraction(oracle.bf16_to_double(int(dec[0, k]))) == want
    with pytest.raises(ValueError):
        oracle.decode_expert_bf16(np.zeros((1, 1, 16), np.uint8), np.full((1, 1, 1), 253, np.uint8), 0)


# ----------------------------------------------------------------- route sort

def test_route_sort_is_stable_argsort():
    rng = np.random.default_rng(3)
    T, k, E = 300, 4, 37
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids[ids == 5] = 6                     # expert 5 empty
    ids[0, :] = 9                         # duplicates within a token are allowed
    gs, off, ss, s2r = oracle.route_sort(ids, E)
    flat = ids.ravel()
    np.testing.assert_array_equal(gs, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    np.testing.assert_array_equal(ss, np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(s2r[ss], np.arange(T * k))
    assert gs[5] == 0
    assert np.all(np.diff(flat[ss]) >= 0)


def test_route_sort_rejects_out_of_range_id():
    with pytest.raises(ValueError):
        oracle.route_sort(np.array([[0, 4]], np.int32), 4)
    with pytest.raises(ValueError):
        oracle.route_sort(np.array([[-1, 0]], np.int32), 4)


def test_route_sort_empty_input():
    gs, off, ss, s2r = oracle.route_sort(np.zeros((0, 6), np.int32), 8)
    assert gs.sum() == 0 and off.tolist() == [0] * 9 and ss.size == 0


def test_gather_copies_token_rows():
    x = np.arange(5 * 3, dtype=np.uint16).reshape(5, 3)
    ss = np.array([4, 0, 9, 2], np.int32)          # slots with k = 2 -> tokens 2, 0, 4, 1
    np.testing.assert_array_equal(oracle.gather(x, ss, 2), x[[2, 0, 4, 1]])


# --------------------------------------------------------------- grouped GEMM

def _decode_formula(codes, scales):
    """Independent dequantisation: piecewise-linear identity over q, times 2^(s-127)."""
    E, N, Kh = codes.shape
    K = 2 * Kh
    nib = np.empty((E, N, K), np.int64)
    nib[..., 0::2] = codes & 15
    nib[..., 1::2] = codes >> 4
    q = np.where(nib & 8, -(nib & 7), nib & 7).astype(np.float64)
    v = 2 * q - np.clip(q, -6, 6) - 0.5 * np.clip(q, -4, 4)
    s = np.repeat(scales.astype(np.int64), 32, axis=2)
    return np.ldexp(v, s - 127)


def test_gemm_tiny_exact_rational():
    rng = np.random.default_rng(4)
    E, N, K = 3, 5, 64
    gs = np.array([2, 0, 3], np.int32)
    rows = int(gs.sum())
    codes = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    scales = rng.integers(117, 126, size=(E, N, K // 32)).astype(np.uint8)
    act = inputs.f32_to_bf16_bits(rng.standard_normal((rows, K)).astype(np.float32))
    out, mag = oracle.grouped_gemm(act, codes, scales, gs, n_threads=2)
    a = inputs.bf16_bits_to_f32(act)
    band = np.repeat(np.arange(E), gs)
    for r in range(rows):
        e = band[r]
        for n in range(N):
            exact = Fraction(0)
            for k in range(K):
                byte = int(codes[e, n, k // 2])
                c = byte & 15 if k % 2 == 0 else byte >> 4
                s, ee, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
                w = Fraction(m, 2) if ee == 0 else Fraction(2) ** (ee - 1) * (1 + Fraction(m, 2))
                w = (-w if s else w) * Fraction(2) ** (int(scales[e, n, k // 32]) - 127)
                exact += Fraction(float(a[r, k])) * w
            assert abs(Fraction(out[r, n]) - exact) <= Fraction(mag[r, n]) * Fraction(K, 2 ** 52)


def test_gemm_single_expert_is_dense_matmul():
    rng = np.random.default_rng(5)
    N, K, rows = 48, 160, 7                      # N != K: a transposed operand fails
    codes = rng.integers(0, 256, size=(1, N, K // 2), dtype=np.uint8)
    scales = rng.integers(100, 140, size=(1, N, K // 32)).astype(np.uint8)
    act = inputs.f32_to_bf16_bits(rng.standard_normal((rows, K)).astype(np.float32))
    out, _ = oracle.grouped_gemm(act, codes, scales, np.array([rows], np.int32))
    ref = inputs.bf16_bits_to_f32(act).astype(np.float64) @ _decode_formula(codes, scales)[0].T
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-300)


def test_gemm_bands_follow_expert_order():
    rng = np.random.default_rng(6)
    E, N, K = 5, 16, 96
    gs = np.array([3, 0, 1, 4, 0], np.int32)
    codes = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    scales = rng.integers(110, 130, size=(E, N, K // 32)).astype(np.uint8)
    act = inputs.f32_to_bf16_bits(rng.standard_normal((8, K)).astype(np.float32))
    out, _ = oracle.grouped_gemm(act, codes, scales, gs)
    W = _decode_formula(codes, scales)
    a = inputs.bf16_bits_to_f32(act).astype(np.float64)
    ref = np.concatenate([a[0:3] @ W[0].T, a[3:4] @ W[2].T, a[4:8] @ W[3].T])
    np.testing.assert_allclose(out, ref, rtol=1e-12)


def test_gemm_nibble_order_and_scale_blocks():
    # act one-hot at k picks column k of the weights.
    K, N = 64, 2
    codes = np.zeros((1, N, K // 2), np.uint8)
    codes[0, 0, 0] = 0x02      # k=0 -> 1.0 (low nibble), k=1 -> 0
    codes[0, 1, 0] = 0x20      # k=0 -> 0, k=1 -> 1.0 (high nibble)
    codes[0, 0, 20] = 0x0C     # k=40 -> -2.0
    scales = np.full((1, N, 2), 127, np.uint8)
    scales[0, 0, 1] = 130      # block 1 (k = 32..63) scaled by 2^3
    one = np.float32(1.0)
    act = np.zeros((3, K), np.uint16)
    act[0, 0] = inputs.f32_to_bf16_bits(np.array([one]))[0]
    act[1, 1] = inputs.f32_to_bf16_bits(np.array([one]))[0]
    act[2, 40] = inputs.f32_to_bf16_bits(np.array([one]))[0]
    out, _ = oracle.grouped_gemm(act, codes, scales, np.array([3], np.int32))
    np.testing.assert_array_equal(out, [[1.0, 0.0], [0.0, 1.0], [-16.0, 0.0]])


def test_gemm_identity_weights_reproduce_activations():
    K = N = 64
    codes = np.zeros((1, N, K // 2), np.uint8)
    for n in range(N):
        codes[0, n, n // 2] = 0x02 if n % 2 == 0 else 0x20    # 1.0 on the diagonal
    scales = np.full((1, N, K // 32), 127, np.uint8)
    rng = np.random.default_rng(7)
    act = inputs.f32_to_bf16_bits(rng.standard_normal((9, K)).astype(np.float32))
    out, _ = oracle.grouped_gemm(act, codes, scales, np.array([9], np.int32))
    np.testing.assert_array_equal(out, inputs.bf16_bits_to_f32(act).astype(np.float64))


def test_gemm_empty_expert_weights_are_never_used():
    case = inputs.gemm_case("tiny", seed=0)
    gs, *_ = oracle.route_sort(case["ids"], case["E"])
    assert gs[5] == 0
    out1, _ = oracle.grouped_gemm(case["act"], case["codes"], case["scales"], gs)
    codes, scales = case["codes"].copy(), case["scales"].copy()
    codes[5] = 0x77
    scales[5] = 0xFE                  # would be rejected if it were read
    out2, _ = oracle.grouped_gemm(case["act"], codes, scales, gs)
    np.testing.assert_array_equal(out1, out2)


def test_gemm_rejects_inconsistent_sizes_and_bad_scales():
    act = np.zeros((4, 32), np.uint16)
    codes = np.zeros((2, 8, 16), np.uint8)
    scales = np.full((2, 8, 1), 127, np.uint8)
    with pytest.raises(ValueError):
        oracle.grouped_gemm(act, codes, scales, np.array([1, 2], np.int32))
    scales[1] = 253
    with pytest.raises(ValueError):
        oracle.grouped_gemm(act, codes, scales, np.array([1, 3], np.int32))


def test_gemm_sampled_matches_full():
    case = inputs.gemm_case(dict(E=6, k=2, T=40, K=128, N=96, exp=(-9, -3)), seed=1)
    gs, *_ = oracle.route_sort(case["ids"], case["E"])
    full, mag = oracle.grouped_gemm(case["act"], case["codes"], case["scales"], gs)
    rng = np.random.default_rng(8)
    r = rng.integers(0, case["rows"], 300)
    c = rng.integers(0, case["N"], 300)
    out, m = oracle.grouped_gemm_sampled(case["act"], case["codes"], case["scales"], gs, r, c)
    np.testing.assert_array_equal(out, full[r, c])
    np.testing.assert_array_equal(m, mag[r, c])


# ------------------------------------------------------- scale block of 512

def test_gemm_block512_tiny_exact_rational():
    # Two 512-k scale blocks per row, scales differing across the boundary;
    # every weight is rebuilt from the OCP bit fields and 2^(s - 127) with the
    # scale indexed by k // 512.
    rng = np.random.default_rng(14)
    E, N, K = 2, 3, 1024
    gs = np.array([2, 1], np.int32)
    rows = int(gs.sum())
    codes = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    scales = rng.integers(120, 134, size=(E, N, K // 512)).astype(np.uint8)
    act = inputs.f32_to_bf16_bits(rng.standard_normal((rows, K)).astype(np.float32))
    out, mag = oracle.grouped_gemm_block(act, codes, scales, gs, 512, n_threads=2)
    a = inputs.bf16_bits_to_f32(act)
    band = np.repeat(np.arange(E), gs)
    for r in range(rows):
        e = band[r]
        for n in range(N):
            exact = Fraction(0)
            for k in range(K):
                byte = int(codes[e, n, k // 2])
                c = byte & 15 if k % 2 == 0 else byte >> 4
                sg, ee, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
                w = Fraction(m, 2) if ee == 0 else Fraction(2) ** (ee - 1) * (1 + Fraction(m, 2))
                w = (-w if sg else w) * Fraction(2) ** (int(scales[e, n, k // 512]) - 127)
                exact += Fraction(float(a[r, k])) * w
            assert abs(Fraction(out[r, n]) - exact) <= Fraction(mag[r, n]) * Fraction(K, 2 ** 52)


def test_gemm_block512_one_hot_at_the_block_boundary():
    # act one-hot at k = 511 and k = 512 picks the last weight of scale block 0
    # and the first of block 1; code 0x2 is 1.0, so the outputs are the scales.
    K, N = 1024, 2
    codes = np.zeros((1, N, K // 2), np.uint8)
    codes[0, :, 255] = 0x20          # k = 511 (high nibble of byte 255)
    codes[0, :, 256] = 0x02          # k = 512 (low nibble of byte 256)
    scales = np.array([[[120, 131], [127, 100]]], np.uint8)
    one = inputs.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    act = np.zeros((2, K), np.uint16)
    act[0, 511] = one
    act[1, 512] = one
    out, _ = oracle.grouped_gemm_block(act, codes, scales, np.array([2], np.int32), 512)
    np.testing.assert_array_equal(out, [[2.0 ** -7, 1.0], [2.0 ** 4, 2.0 ** -27]])


def test_gemm_block512_equals_block32_with_repeated_scales():
    # A 512-block scale is the same scale on each of its sixteen 32-blocks, so
    # the result must equal the (separately pinned) block-32 GEMM bit for bit.
    case = inputs.gemm_case(dict(E=5, k=2, T=30, K=1024, N=64, exp=(-9, -3)), seed=3)
    gs, *_ = oracle.route_sort(case["ids"], case["E"])
    rng = np.random.default_rng(15)
    s512 = rng.integers(115, 131, size=(case["E"], case["N"], case["K"] // 512)).astype(np.uint8)
    out512, mag512 = oracle.grouped_gemm_block(case["act"], case["codes"], s512, gs, 512)
    out32, mag32 = oracle.grouped_gemm(case["act"], case["codes"], np.repeat(s512, 16, axis=2), gs)
    np.testing.assert_array_equal(out512, out32)
    np.testing.assert_array_equal(mag512, mag32)
    # block 32 through the block entry point is the block-32 GEMM itself
    o32, _ = oracle.grouped_gemm_block(case["act"], case["codes"], case["scales"], gs, 32)
    np.testing.assert_array_equal(o32, oracle.grouped_gemm(case["act"], case["codes"], case["scales"], gs)[0])


def test_gemm_block_rejects_other_blocks_and_ragged_k():
    act = np.zeros((2, 512), np.uint16)
    codes = np.zeros((1, 8, 256), np.uint8)
    with pytest.raises(ValueError):
        oracle.grouped_gemm_block(act, codes, np.full((1, 8, 8), 127, np.uint8), np.array([2], np.int32), 64)
    act = np.zeros((2, 768), np.uint16)
    codes = np.zeros((1, 8, 384), np.uint8)
    with pytest.raises(ValueError):      # K = 768 is not a multiple of 512
        oracle.grouped_gemm_block(act, codes, np.full((1, 8, 2), 127, np.uint8), np.array([2], np.int32), 512)


# --------------------------------------------------------------------- SwiGLU

def test_swiglu_closed_forms():
    # I = 2: columns [g0, g1, u0, u1].  g = 0 gives 0 whatever u; u = 0 gives
    # (signed) 0 whatever g; g = u = 0 gives +0.
    gu = np.array([[0.0, 1.0, 5.0, 0.0],
                   [3.0, 0.0, 0.0, -7.0]])
    h = oracle.swiglu(gu)
    assert h[0, 0] == 0 and h[0, 1] & 0x7FFF == 0 and h[1, 0] & 0x7FFF == 0 and h[1, 1] & 0x7FFF == 0
    # silu(g) - silu(-g) = g; with u = 1 both sides are rounded once to bf16.
    for g in (0.25, 1.0, 2.5, 7.0):
        hp = oracle.bf16_to_double(int(oracle.swiglu(np.array([[g, 1.0]]))[0, 0]))
        hm = oracle.bf16_to_double(int(oracle.swiglu(np.array([[-g, 1.0]]))[0, 0]))
        assert abs((hp - hm) - g) <= 2 ** -8 * (abs(hp) + abs(hm))


def test_swiglu_matches_logistic_library_routine():
    special = pytest.importorskip("scipy.special")
    gu = inputs.gate_up_f32(9, 64, 48).astype(np.float64)
    h = oracle.swiglu(gu)
    g, u = gu[:, :48], gu[:, 48:]
    ref = np.array([[oracle.double_to_bf16(v) for v in row] for row in g * special.expit(g) * u],
                   dtype=np.uint16)
    diff = np.abs(h.astype(np.int64) - ref.astype(np.int64))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.999


# -------------------------------------------------------------------- combine

def test_combine_unpermutes_with_unit_weight():
    rng = np.random.default_rng(10)
    T, N = 11, 7
    y = rng.standard_normal((T, N))
    perm = rng.permutation(T).astype(np.int32)
    out, _ = oracle.combine(y, perm, np.ones((T, 1), np.float32))
    np.testing.assert_array_equal(out, y[perm])


def test_combine_matches_einsum():
    rng = np.random.default_rng(11)
    T, k, N = 13, 3, 10
    y = rng.standard_normal((T * k, N))
    s2r = rng.permutation(T * k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    out, mag = oracle.combine(y, s2r, w)
    ref = np.einsum("tj,tjn->tn", w.astype(np.float64), y[s2r].reshape(T, k, N))
    np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(mag, np.einsum("tj,tjn->tn", np.abs(w), np.abs(y[s2r].reshape(T, k, N))),
                               rtol=1e-14)


# ------------------------------------------------------- composed layer (E=1)

def test_single_expert_layer_is_dense_swiglu_mlp():
    special = pytest.importorskip("scipy.special")
    c = inputs.layer_case(seed=2, T=5, E=1, hidden=64, inter=32, k=1)
    gs, off, ss, s2r = oracle.route_sort(c["ids"], 1)
    xs = oracle.gather(c["x"], ss, 1)
    y13, _ = oracle.grouped_gemm(xs, c["w13_codes"], c["w13_scales"], gs)
    h = oracle.swiglu(y13)
    y2, _ = oracle.grouped_gemm(h, c["w2_codes"], c["w2_scales"], gs)
    out, _ = oracle.combine(y2, s2r, c["topk_w"])
    x = inputs.bf16_bits_to_f32(c["x"]).astype(np.float64)
    W13 = _decode_formula(c["w13_codes"], c["w13_scales"])[0]
    W2 = _decode_formula(c["w2_codes"], c["w2_scales"])[0]
    g13 = x @ W13.T
    hh = g13[:, :32] * special.expit(g13[:, :32]) * g13[:, 32:]
    hb = np.array([[oracle.double_to_bf16(v) for v in row] for row in hh], dtype=np.uint16)
    assert np.abs(h.astype(np.int64) - hb.astype(np.int64)).max() <= 1
    hd = inputs.bf16_bits_to_f32(h).astype(np.float64)
    ref = (hd @ W2.T) * c["topk_w"].astype(np.float64)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-300)


# ------------------------------------------- MXFP4 -> NVFP4 lossless weight cast
# "DeepSeek-V4-Flash-0731-NVFP4", "The lossless weight cast": the per-tensor
# scale is 2^(k_max - 8) and every per-16 E4M3 scale 2^(k_j - k_max + 8), with
# the 4-bit codes unchanged, so the dequantized weights are identical.

def test_e4m3_value_matches_torch_float8_for_every_byte():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(b) for b in range(256)])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_e4m3_anchor_values():
    # the format's definition: 0x38 = 1, 0x78 = 2^8, 0x7E = 448 (largest),
    # 0x08 = 2^-6 (smallest normal), 0x01 = 2^-9 (smallest subnormal), 0xB8 = -1
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0x78) == 256.0
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_value(0x7F))


def _dequant_mxfp4(codes, scales):
    E, N, Kh = codes.shape
    lo, hi = codes & 15, codes >> 4
    q = np.empty((E, N, 2 * Kh), np.int64)
    q[..., 0::2], q[..., 1::2] = lo, hi
    vals = np.array([oracle.e2m1_value(c) for c in range(16)])[q]
    return vals * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=2)


def _dequant_nvfp4(codes, e4m3, ws2):
    E, N, Kh = codes.shape
    lo, hi = codes & 15, codes >> 4
    q = np.empty((E, N, 2 * Kh), np.int64)
    q[..., 0::2], q[..., 1::2] = lo, hi
    vals = np.array([oracle.e2m1_value(c) for c in range(16)])[q]
    s16 = np.array([oracle.e4m3_value(b) for b in range(256)])[e4m3]
    return vals * np.repeat(s16, 16, axis=2) * ws2[:, None, None]


def test_cast_dequantizes_to_identical_values_when_in_range():
    rng = np.random.default_rng(21)
    E, N, K = 3, 8, 256
    codes = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    top = np.array([127 + 40, 127 - 60, 200])[:, None, None]
    scales = (top - rng.integers(0, 18, (E, N, K // 32))).astype(np.uint8)   # spread <= 17
    e4m3, ws2, oob = oracle.mxfp4_to_nvfp4(scales)
    assert (oob == 0).all()
    assert np.array_equal(_dequant_nvfp4(codes, e4m3, ws2), _dequant_mxfp4(codes, scales))


def test_cast_closed_forms_at_the_edges_of_the_range():
    s = np.array([[[130, 130 - 17, 130 - 18, 130 - 5]]], np.uint8)   # k_max = 3
    e4m3, ws2, oob = oracle.mxfp4_to_nvfp4(s)
    assert ws2[0] == 2.0 ** (3 - 8)
    assert list(e4m3[0, 0]) == [0x78, 0x78, 0x01, 0x01, 0, 0, 0x50, 0x50]   # 2^8, 2^-9, -, 2^3
    assert oob[0] == 1


def test_cast_out_of_range_count_is_brute_force():
    rng = np.random.default_rng(22)
    s = rng.integers(0, 255, (4, 16, 8), dtype=np.uint8)
    _, ws2, oob = oracle.mxfp4_to_nvfp4(s)
    for e in range(4):
        k = s[e].astype(np.int64) - 127
        assert oob[e] == int((k < k.max() - 17).sum())
        assert ws2[e] == 2.0 ** (k.max() - 8)


def test_cast_shares_k_max_across_the_fused_rows_and_rejects_nan_scale():
    # rows [0, I) (w1) small, rows [I, 2I) (w3) large: one k_max for the tensor
    s = np.full((1, 4, 2), 120, np.uint8)
    s[0, 2:] = 125
    _, ws2, _ = oracle.mxfp4_to_nvfp4(s)
    assert ws2[0] == 2.0 ** (125 - 127 - 8)
    s[0, 0, 0] = 255
    with pytest.raises(ValueError):
        oracle.mxfp4_to_nvfp4(s)


# ------------------------------------------------------------ NVFP4 grouped GEMM
# "Running DeepSeek V4 Flash on TPU v6", section 1: an NVFP4 kernel decodes the
# e2m1 weights and their per-16 E4M3 scales; "DeepSeek-V4-Flash-0731-NVFP4",
# "The lossless weight cast": the per-16 E4M3 scale and the per-tensor
# weight_scale_2 together reconstruct each weight.  The pins decode E4M3 with
# torch's float8_e4m3fn and e2m1 from the page's magnitudes, not the oracle.

def _torch_e4m3(bytes_):
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    t = torch.from_numpy(np.ascontiguousarray(bytes_, np.uint8).reshape(-1)).view(torch.float8_e4m3fn)
    return t.double().numpy().reshape(np.shape(bytes_))


def _e2m1_from_page(codes, mags):
    E, N, Kh = codes.shape
    q = np.empty((E, N, 2 * Kh), np.int64)
    q[..., 0::2], q[..., 1::2] = codes & 15, codes >> 4
    mag = np.asarray(mags, np.float64)[q & 7]
    return np.where(q & 8, -mag, mag)


def _random_e4m3_scales(rng, shape, lo=0x20, hi=0x58):
    """Finite E4M3 bytes with random mantissas and both signs (0x7F/0xFF excluded)."""
    b = rng.integers(lo, hi, size=shape).astype(np.uint8)
    return b | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)


def test_nvfp4_gemm_tiny_exact_rational(golden_dir):
    rng = np.random.default_rng(31)
    mags = _golden_magnitudes(golden_dir)
    E, N, K = 3, 5, 64
    gs = np.array([2, 0, 3], np.int32)
    rows = int(gs.sum())
    codes = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    s16 = _random_e4m3_scales(rng, (E, N, K // 16))
    ws2 = (np.float32(2.0) ** rng.integers(-12, 4, E) * (1 + rng.integers(0, 8, E) / 8)).astype(np.float32)
    act = inputs.f32_to_bf16_bits(rng.standard_normal((rows, K)).astype(np.float32))
    out, mag = oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, gs, n_threads=2)
    a = inputs.bf16_bits_to_f32(act)
    w2 = _e2m1_from_page(codes, mags)
    sv = _torch_e4m3(s16)
    band = np.repeat(np.arange(E), gs)
    for r in range(rows):
        e = band[r]
        for n in range(N):
            exact = Fraction(0)
            for k in range(K):
                w = Fraction(float(w2[e, n, k])) * Fraction(float(sv[e, n, k // 16])) * Fraction(float(ws2[e]))
                exact += Fraction(float(a[r, k])) * w
            assert abs(Fraction(out[r, n]) - exact) <= Fraction(mag[r, n]) * Fraction(K, 2 ** 52)


def test_nvfp4_gemm_single_expert_is_dense_matmul(golden_dir):
    rng = np.random.default_rng(32)
    N, K, rows = 48, 160, 7                      # N != K: a transposed operand fails
    codes = rng.integers(0, 256, size=(1, N, K // 2), dtype=np.uint8)
    s16 = _random_e4m3_scales(rng, (1, N, K // 16))
    ws2 = np.array([0.0625 * 1.375], np.float32)
    act = inputs.f32_to_bf16_bits(rng.standard_normal((rows, K)).astype(np.float32))
    out, _ = oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, np.array([rows], np.int32))
    W = _e2m1_from_page(codes, _golden_magnitudes(golden_dir)) * np.repeat(_torch_e4m3(s16), 16, axis=2)
    ref = inputs.bf16_bits_to_f32(act).astype(np.float64) @ (W[0] * float(ws2[0])).T
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-300)


def test_nvfp4_scale_blocks_are_16_wide_and_tensor_scale_per_expert():
    # act one-hot at k picks column k: k = 15 and k = 16 fall in different
    # per-16 blocks; expert 1 has its own per-tensor scale.
    K, N = 32, 1
    codes = np.full((2, N, K // 2), 0x22, np.uint8)        # every weight code 1.0
    s16 = np.zeros((2, N, 2), np.uint8)
    s16[:, 0, 0] = 0x38                                    # block 0: 1.0
    s16[:, 0, 1] = 0x44                                    # block 1: 1.5 * 2 = 3.0
    ws2 = np.array([0.5, 4.0], np.float32)
    one = inputs.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    act = np.zeros((4, K), np.uint16)
    act[0, 15] = act[1, 16] = act[2, 15] = act[3, 16] = one
    out, _ = oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, np.array([2, 2], np.int32))
    np.testing.assert_array_equal(out[:, 0], [0.5, 1.5, 4.0, 12.0])


def test_nvfp4_gemm_of_the_lossless_cast_equals_the_mxfp4_gemm():
    # MXFP4 weights cast losslessly to NVFP4 reconstruct the same values, so
    # both GEMMs sum identical exact products in the same order.
    case = inputs.gemm_case(dict(E=6, k=2, T=40, K=128, N=96, exp=(-9, -3)), seed=3)
    gs, *_ = oracle.route_sort(case["ids"], case["E"])
    mx, mx_mag = oracle.grouped_gemm(case["act"], case["codes"], case["scales"], gs)
    e4m3, ws2, oob = oracle.mxfp4_to_nvfp4(case["scales"])
    assert (oob == 0).all()
    nv, nv_mag = oracle.nvfp4_grouped_gemm(case["act"], case["codes"], e4m3, ws2.astype(np.float32), gs)
    np.testing.assert_array_equal(nv, mx)
    np.testing.assert_array_equal(nv_mag, mx_mag)


def test_nvfp4_gemm_rejects_nan_scales_and_bad_sizes_but_never_reads_empty_experts():
    act = np.zeros((4, 32), np.uint16)
    codes = np.zeros((2, 8, 16), np.uint8)
    s16 = np.full((2, 8, 2), 0x38, np.uint8)
    ws2 = np.ones(2, np.float32)
    s16[1, 3, 1] = 0x7F                                    # E4M3 NaN in expert 1
    oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, np.array([4, 0], np.int32))   # expert 1 empty
    with pytest.raises(ValueError):
        oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, np.array([1, 3], np.int32))
    s16[1, 3, 1] = 0xFF
    with pytest.raises(ValueError):
        oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, np.array([2, 2], np.int32))
    with pytest.raises(ValueError):                        # rows != sum(group_sizes)
        oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, np.array([1, 0], np.int32))
    with pytest.raises(ValueError):                        # K % 16
        oracle.nvfp4_grouped_gemm(np.zeros((1, 24), np.uint16), np.zeros((1, 8, 12), np.uint8),
                                  np.full((1, 8, 1), 0x38, np.uint8), ws2[:1], np.array([1], np.int32))
