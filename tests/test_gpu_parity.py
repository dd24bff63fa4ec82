"""GPU parity: every kernel, called through the C ABI, against the CPU oracle on
the same seeded inputs.

Bars: route sort, gather and decoded weights bit-exact; GEMM f32 outputs within
|gpu - oracle| <= 1e-5 * sum_k |a_k w_k| + 1e-6 per element (bf16 outputs: one
bf16 ulp more); SwiGLU within 1 bf16 ulp of the oracle fed the GPU's input;
combine within 1e-6 * sum_j |w_j y_j| + 1e-6; every kernel bitwise repeatable.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_weight_grouped_gb300 import inputs
from parity_bounds import check_swiglu_from_gemm

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as g
    g.build()
    from fp4_weight_grouped_gb300 import binding
    binding.load()
    return binding


def _tol_check(gpu, ref, mag, rel=1e-5, abs_=1e-6, extra=None, what=""):
    gpu = np.asarray(gpu, np.float64)
    bound = rel * mag + abs_
    if extra is not None:
        bound = bound + extra
    diff = np.abs(gpu - ref)
    bad = ~(diff <= bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {diff.size} outside tolerance; "
                           f"worst ratio {float(np.max(diff / bound)):.3g}")
    return float(np.max(diff / bound)) if diff.size else 0.0


def k8_interleave(a):
    """Natural k order -> the K8-interleaved order [0,4,1,5,2,6,3,7] per group of 8."""
    a = np.ascontiguousarray(a)
    K = a.shape[-1]
    return a.reshape(*a.shape[:-1], K // 8, 2, 4).swapaxes(-1, -2).reshape(a.shape)


def k8_deinterleave(a):
    a = np.ascontiguousarray(a)
    K = a.shape[-1]
    return a.reshape(*a.shape[:-1], K // 8, 4, 2).swapaxes(-1, -2).reshape(a.shape)


def test_k8_helpers_are_inverse_and_match_header_order():
    a = np.arange(16).reshape(1, 16)
    assert k8_interleave(a).tolist() == [[0, 4, 1, 5, 2, 6, 3, 7, 8, 12, 9, 13, 10, 14, 11, 15]]
    np.testing.assert_array_equal(k8_deinterleave(k8_interleave(a)), a)


def _bf16_ulp(x):
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    return np.ldexp(1.0, (np.maximum(e, -126) - 7).astype(np.int64))


def _gemm_gpu(B, act, codes, scales, gs, out_dtype=torch.float32, k8=False):
    ws = B.make_workspace(0, 1, 1, DEV)
    a = k8_interleave(act) if k8 else act
    out = B.grouped_gemm(B.bf16_from_bits(a, DEV), B.to_device(codes, DEV), B.to_device(scales, DEV),
                         B.to_device(np.asarray(gs, np.int32), DEV), out_dtype=out_dtype, workspace=ws,
                         act_layout=B.MOE_ACT_K8_INTERLEAVED if k8 else B.MOE_ACT_ROW_MAJOR)
    st = B.read_status(ws)
    assert st == B.MOE_OK, B.status_string(st)
    if out_dtype == torch.bfloat16:
        return B.bits_from_bf16(out)
    return out.cpu().numpy()


# ------------------------------------------------------------------ route sort

ROUTE_CASES = [
    ("tiny", lambda: (inputs.gemm_case("tiny")["ids"], 8)),
    ("decode_w13", lambda: (inputs.route_uniform(0, 64, 256, 6), 256)),
    ("decode_w2", lambda: (inputs.route_uniform(0, 256, 256, 6), 256)),
    ("prefill_zipf", lambda: (inputs.route_zipf(0, 4096, 256, 6), 256)),
    ("layer", lambda: (inputs.route_logits(0, 8192, 256, 6)[0], 256)),
    ("one_expert", lambda: (np.zeros((37, 1), np.int32), 1)),
    ("dup_and_wide", lambda: (np.random.default_rng(5).integers(0, 1024, (3001, 3)).astype(np.int32), 1024)),
    ("empty", lambda: (np.zeros((0, 6), np.int32), 16)),
]


@pytest.mark.parametrize("k8", [False, True], ids=["row_major", "k8"])
@pytest.mark.parametrize("name,make", ROUTE_CASES, ids=[c[0] for c in ROUTE_CASES])
def test_route_sort_bit_exact(B, name, make, k8):
    ids, E = make()
    T, k = ids.shape
    hidden = 64
    x = inputs.normal_bf16(1, 99, (T, hidden))
    ws = B.make_workspace(T, k, E, DEV)
    gs, off, ss, s2r, xs = B.route_sort(B.to_device(ids, DEV), E, B.bf16_from_bits(x, DEV), ws,
                                        x_layout=B.MOE_ACT_K8_INTERLEAVED if k8 else B.MOE_ACT_ROW_MAJOR)
    assert B.read_status(ws) == B.MOE_OK
    o_gs, o_off, o_ss, o_s2r = oracle.route_sort(ids, E)
    np.testing.assert_array_equal(gs.cpu().numpy(), o_gs)
    np.testing.assert_array_equal(off.cpu().numpy(), o_off)
    np.testing.assert_array_equal(ss.cpu().numpy(), o_ss)
    np.testing.assert_array_equal(s2r.cpu().numpy(), o_s2r)
    got = B.bits_from_bf16(xs)
    np.testing.assert_array_equal(k8_deinterleave(got) if k8 else got, oracle.gather(x, o_ss, k))


def test_route_sort_repeatable_and_flags_bad_ids(B):
    ids = inputs.route_logits(3, 2048, 256, 6)[0]
    dids = B.to_device(ids, DEV)
    a = [t.clone() for t in B.route_sort(dids, 256)[:4]]
    b = B.route_sort(dids, 256)[:4]
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    bad = ids.copy()
    bad[100, 3] = 256
    ws = B.make_workspace(*bad.shape, 256, DEV)
    B.route_sort(B.to_device(bad, DEV), 256, workspace=ws)
    assert B.read_status(ws) == B.MOE_ERR_DATA


# -------------------------------------------------------------- weight decode

def test_decode_bit_exact_all_codes_and_scale_edges(B):
    rng = np.random.default_rng(7)
    E, N, K = 2, 256, 512
    codes = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    codes[1, :, :128] = np.arange(256, dtype=np.uint8)[None, :128].repeat(N, 0)
    codes[1, :, 128:] = np.arange(128, 256, dtype=np.uint8)[None, :].repeat(N, 0)
    scales = rng.integers(0, 253, (E, N, K // 32), dtype=np.uint8)
    scales[1, :8, :] = np.array([0, 1, 2, 3, 126, 127, 251, 252], np.uint8)[:, None]
    for e in range(E):
        got = B.bits_from_bf16(B.decode_expert(B.to_device(codes, DEV), B.to_device(scales, DEV), e))
        np.testing.assert_array_equal(got, oracle.decode_expert_bf16(codes, scales, e))


def test_decode_flags_out_of_range_scale(B):
    codes = np.full((1, 16, 32), 0x22, np.uint8)
    scales = np.full((1, 16, 2), 127, np.uint8)
    scales[0, 3, 1] = 253
    ws = B.make_workspace(0, 1, 1, DEV)
    out = B.decode_expert(B.to_device(codes, DEV), B.to_device(scales, DEV), 0, workspace=ws)
    assert B.read_status(ws) == B.MOE_ERR_DATA
    assert torch.isnan(out[3, 32:].float()).all() and not torch.isnan(out[3, :32].float()).any()


@pytest.mark.parametrize("scale_range", [(2, 128), (2, 252), (120, 135)],
                         ids=["one_fma_path", "split_path", "path_boundary"])
@pytest.mark.parametrize("k8", [False, True], ids=["row_major", "k8"])
def test_gemm_identity_activations_expose_decoded_weights(B, scale_range, k8):
    # act = I_K: out[k, n] = w[n, k] exactly, so the converter's decode is checked
    # bit for bit inside the GEMM.  Scale bytes >= 2 keep every weight an f32
    # normal number (subnormal products may be flushed by the tensor pipe; the
    # decode entry point covers scale bytes 0 and 1 bit for bit).
    rng = np.random.default_rng(8)
    K, N = 256, 384
    codes = rng.integers(0, 256, (1, N, K // 2), dtype=np.uint8)
    scales = rng.integers(scale_range[0], scale_range[1] + 1, (1, N, K // 32), dtype=np.uint8)
    one = inputs.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    act = np.zeros((K, K), np.uint16)
    act[np.arange(K), np.arange(K)] = one
    out = _gemm_gpu(B, act, codes, scales, [K], k8=k8)
    dec = inputs.bf16_bits_to_f32(oracle.decode_expert_bf16(codes, scales, 0))
    np.testing.assert_array_equal(out, dec.T)


@pytest.mark.parametrize("rows", [32, 16], ids=["bands32", "bands16"])
@pytest.mark.parametrize("scale_range", [(2, 128), (2, 252)], ids=["one_fma_path", "split_path"])
def test_gemm_split_mode_exposes_decoded_weights(B, scale_range, rows):
    # 512 // rows experts x `rows` rows, K = 512: row r of expert e is one-hot at
    # k = rows * e + r, so out[row, n] = w_e[n, rows * e + r] exactly.  Bands of
    # <= 32 rows select the split-accumulator mode, <= 16 its narrow layout.
    rng = np.random.default_rng(9)
    K, N = 512, 256
    E = K // rows
    codes = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    scales = rng.integers(scale_range[0], scale_range[1] + 1, (E, N, K // 32), dtype=np.uint8)
    one = inputs.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    act = np.zeros((K, K), np.uint16)
    act[np.arange(K), np.arange(K)] = one
    out = _gemm_gpu(B, act, codes, scales, np.full(E, rows, np.int32))
    for e in range(E):
        dec = inputs.bf16_bits_to_f32(oracle.decode_expert_bf16(codes, scales, e))
        np.testing.assert_array_equal(out[rows * e:rows * e + rows],
                                      dec[:, rows * e:rows * e + rows].T)


# ---------------------------------------------------------------- grouped GEMM

def _explicit(gs, K, N, E=None, seed=0, exp=(-9, -3)):
    gs = np.asarray(gs, np.int32)
    E = len(gs) if E is None else E
    act = inputs.normal_bf16(seed, 11, (int(gs.sum()), K))
    codes, scales = inputs.mxfp4_weights(seed, 12, E, N, K, exp)
    return act, codes, scales, gs


GEMM_CASES = {
    # bands of every shape class: empty, 1 row, around 16, around 128, > 2 chunks
    "ragged_bands": lambda: _explicit([0, 1, 15, 16, 17, 127, 128, 129, 300, 0, 5], 512, 256),
    # K not a multiple of the 128-wide stage, N not a multiple of the 128-wide tile
    "k_tail_96": lambda: _explicit([9, 0, 33], 96, 200),
    "k_tail_160": lambda: _explicit([40, 3], 160, 136),
    "k_tail_224": lambda: _explicit([1, 2, 250], 224, 72),
    "few_rows": lambda: _explicit([3, 0, 2], 256, 128),
    "one_expert_long_band": lambda: _explicit([700], 256, 128),
    "many_items": lambda: _explicit(np.random.default_rng(3).integers(0, 40, 64), 512, 512),
    # every band <= 32 rows: the split-accumulator mode
    "split_small_bands": lambda: _explicit([0, 1, 7, 16, 0, 3, 32, 12, 17, 31], 1024, 384),
    "split_k_tail_640": lambda: _explicit([5, 0, 16, 9], 640, 200),      # last 64-k stages all zero
    "split_k_tail_544": lambda: _explicit([2, 11, 0, 30], 544, 136),     # K/32 = 17 scale bytes per row
    "split_k_96": lambda: _explicit([3, 0, 8], 96, 128),                 # one partial code stage
    "split_one_row_experts": lambda: _explicit(np.ones(40, np.int32), 2048, 256),
    # the largest expert count: 1024 experts, 300 of them with one row, the rest empty
    "max_experts_sparse": lambda: _explicit(
        np.isin(np.arange(1024), np.random.default_rng(4).choice(1024, 300, replace=False))
        .astype(np.int32), 256, 128),
}


@pytest.mark.parametrize("k8", [False, True], ids=["row_major", "k8"])
@pytest.mark.parametrize("name", sorted(GEMM_CASES))
def test_gemm_matches_oracle(B, name, k8):
    act, codes, scales, gs = GEMM_CASES[name]()
    out = _gemm_gpu(B, act, codes, scales, gs, k8=k8)
    ref, mag = oracle.grouped_gemm(act, codes, scales, gs)
    _tol_check(out, ref, mag, what=name)


def test_gemm_tiny_config(B):
    c = inputs.gemm_case("tiny")
    gs, *_ = oracle.route_sort(c["ids"], c["E"])
    g_gs = B.route_sort(B.to_device(c["ids"], DEV), c["E"])[0]
    np.testing.assert_array_equal(g_gs.cpu().numpy(), gs)
    assert gs[5] == 0
    out = _gemm_gpu(B, c["act"], c["codes"], c["scales"], gs)
    ref, mag = oracle.grouped_gemm(c["act"], c["codes"], c["scales"], gs)
    _tol_check(out, ref, mag, what="tiny")


def test_gemm_bf16_output(B):
    act, codes, scales, gs = _explicit([5, 0, 130, 17], 384, 256)
    out = inputs.bf16_bits_to_f32(_gemm_gpu(B, act, codes, scales, gs, torch.bfloat16))
    ref, mag = oracle.grouped_gemm(act, codes, scales, gs)
    _tol_check(out, ref, mag, extra=_bf16_ulp(ref), what="bf16 out")


def test_gemm_empty_experts_are_not_read(B):
    c = inputs.gemm_case("tiny")
    gs, *_ = oracle.route_sort(c["ids"], c["E"])
    base = _gemm_gpu(B, c["act"], c["codes"], c["scales"], gs)
    codes, scales = c["codes"].copy(), c["scales"].copy()
    codes[5] = 0x77
    scales[5] = 0xFE                 # would flag MOE_ERR_DATA if it were decoded
    poisoned = _gemm_gpu(B, c["act"], codes, scales, gs)
    np.testing.assert_array_equal(base, poisoned)


def test_gemm_repeatable(B):
    act, codes, scales, gs = GEMM_CASES["many_items"]()
    a = _gemm_gpu(B, act, codes, scales, gs)
    b = _gemm_gpu(B, act, codes, scales, gs)
    np.testing.assert_array_equal(a, b)


def test_gemm_flags_inconsistent_group_sizes(B):
    act, codes, scales, gs = _explicit([4, 4], 128, 128)
    ws = B.make_workspace(0, 1, 1, DEV)
    out = torch.full((8, 128), float("nan"), device=DEV)
    bad = B.to_device(np.array([4, 5], np.int32), DEV)
    B.grouped_gemm(B.bf16_from_bits(act, DEV), B.to_device(codes, DEV), B.to_device(scales, DEV), bad,
                   out=out, workspace=ws)
    assert B.read_status(ws) == B.MOE_ERR_DATA
    assert torch.isnan(out).all()


@pytest.mark.parametrize("K", [128, 512], ids=["scales_ldg", "scales_tma"])
def test_gemm_flags_out_of_range_scale(B, K):
    act, codes, scales, gs = _explicit([20], K, 128)
    scales[0, 7, 2] = 255
    ws = B.make_workspace(0, 1, 1, DEV)
    B.grouped_gemm(B.bf16_from_bits(act, DEV), B.to_device(codes, DEV), B.to_device(scales, DEV),
                   B.to_device(gs, DEV), workspace=ws)
    assert B.read_status(ws) == B.MOE_ERR_DATA


@pytest.mark.parametrize("K", [256, 1024], ids=["scales_ldg", "scales_tma"])
def test_gemm_ignores_scales_of_rows_beyond_n(B, K):
    # N = 72: the 128-row weight tile of expert 0 also spans rows of expert 1,
    # which is empty and carries out-of-range scale bytes.  Those rows are not
    # part of any output, so no error may be flagged and expert 0 stays exact.
    act, codes, scales, gs = _explicit([9, 0], K, 72)
    scales[1] = 255
    ws = B.make_workspace(0, 1, 1, DEV)
    out = B.grouped_gemm(B.bf16_from_bits(act, DEV), B.to_device(codes, DEV), B.to_device(scales, DEV),
                         B.to_device(gs, DEV), workspace=ws)
    assert B.read_status(ws) == B.MOE_OK
    ref, mag = oracle.grouped_gemm(act, codes, scales, gs)
    _tol_check(out.cpu().numpy(), ref, mag, what="rows beyond N")


@pytest.mark.parametrize("offset", [1, 4], ids=["byte_aligned", "word_aligned"])
@pytest.mark.parametrize("bands", [[5, 0, 9], [40, 3, 70]], ids=["split_mode", "single_mode"])
def test_gemm_scales_at_unaligned_address(B, offset, bands):
    # K = 512 would take the TMA scale path; a scale tensor that does not start
    # on a 16-byte boundary must fall back to per-thread loads and still match.
    act, codes, scales, gs = _explicit(bands, 512, 128)
    backing = torch.zeros(scales.size + 64, dtype=torch.uint8, device=DEV)
    d_scales = backing[offset:offset + scales.size].view(scales.shape)
    d_scales.copy_(torch.from_numpy(scales).to(DEV))
    assert d_scales.data_ptr() % 16 == offset
    ws = B.make_workspace(0, 1, 1, DEV)
    out = B.grouped_gemm(B.bf16_from_bits(act, DEV), B.to_device(codes, DEV), d_scales,
                         B.to_device(gs, DEV), workspace=ws)
    assert B.read_status(ws) == B.MOE_OK
    ref, mag = oracle.grouped_gemm(act, codes, scales, gs)
    _tol_check(out.cpu().numpy(), ref, mag, what=f"scales at +{offset}")


def _sample_pairs(gs, N, n=3000, seed=0):
    """(row, col) samples: random ones plus the first and last row of every band
    and the first and last column."""
    rng = np.random.default_rng(seed)
    rows = int(np.sum(gs))
    off = np.concatenate([[0], np.cumsum(gs)])
    ne = np.nonzero(gs)[0]
    edge_r = np.concatenate([off[ne], off[ne + 1] - 1])
    r = np.concatenate([rng.integers(0, rows, n), edge_r, edge_r])
    c = np.concatenate([rng.integers(0, N, n), rng.integers(0, N, edge_r.size), np.full(edge_r.size, N - 1)])
    return r.astype(np.int64), c.astype(np.int64)


@pytest.mark.parametrize("name", ["decode_w13", "decode_w2", "prefill_w13"])
def test_gemm_full_size_sampled(B, name):
    c = inputs.gemm_case(name)
    gs, *_ = oracle.route_sort(c["ids"], c["E"])
    g_gs = B.route_sort(B.to_device(c["ids"], DEV), c["E"])[0]
    np.testing.assert_array_equal(g_gs.cpu().numpy(), gs)
    out = _gemm_gpu(B, c["act"], c["codes"], c["scales"], gs)
    r, col = _sample_pairs(gs, c["N"])
    ref, mag = oracle.grouped_gemm_sampled(c["act"], c["codes"], c["scales"], gs, r, col)
    _tol_check(out[r, col], ref, mag, what=name)
    assert np.isfinite(out).all()


def test_layer_size_gemms_sampled(B):
    c = inputs.layer_case(seed=0)
    gs, off, ss, s2r = oracle.route_sort(c["ids"], c["E"])
    dev_ids = B.to_device(c["ids"], DEV)
    x = B.bf16_from_bits(c["x"], DEV)
    g_gs, _, g_ss, _, xs = B.route_sort(dev_ids, c["E"], x)
    np.testing.assert_array_equal(g_ss.cpu().numpy(), ss)
    xs_bits = B.bits_from_bf16(xs)
    ws = B.make_workspace(0, 1, 1, DEV)
    y13 = B.grouped_gemm(xs, B.to_device(c["w13_codes"], DEV), B.to_device(c["w13_scales"], DEV), g_gs,
                         workspace=ws)
    r, col = _sample_pairs(gs, 2 * c["inter"], seed=1)
    ref, mag = oracle.grouped_gemm_sampled(xs_bits, c["w13_codes"], c["w13_scales"], gs, r, col)
    _tol_check(y13.cpu().numpy()[r, col], ref, mag, what="layer w13")
    h = B.swiglu(y13)
    y2 = B.grouped_gemm(h, B.to_device(c["w2_codes"], DEV), B.to_device(c["w2_scales"], DEV), g_gs,
                        workspace=ws)
    assert B.read_status(ws) == B.MOE_OK
    r, col = _sample_pairs(gs, c["hidden"], seed=2)
    ref, mag = oracle.grouped_gemm_sampled(B.bits_from_bf16(h), c["w2_codes"], c["w2_scales"], gs, r, col)
    _tol_check(y2.cpu().numpy()[r, col], ref, mag, what="layer w2")


# ------------------------------------------------------------ SwiGLU, combine

@pytest.mark.parametrize("dtype,I,k8", [(torch.float32, 2048, False), (torch.bfloat16, 512, False),
                                        (torch.float32, 40, False), (torch.bfloat16, 12, False),
                                        (torch.float32, 2048, True), (torch.bfloat16, 64, True)])
def test_swiglu_within_one_ulp(B, dtype, I, k8):
    gu = inputs.gate_up_f32(4, 300, I)
    gu[0, :4] = [0.0, -100.0, 95.0, -88.7]
    t = torch.from_numpy(gu).to(DEV).to(dtype)
    h = B.bits_from_bf16(B.swiglu(t, layout=B.MOE_ACT_K8_INTERLEAVED if k8 else B.MOE_ACT_ROW_MAJOR))
    if k8:
        h = k8_deinterleave(h)
    ref = oracle.swiglu(t.float().cpu().numpy().astype(np.float64))
    assert np.abs(h.astype(np.int64) - ref.astype(np.int64)).max() <= 1


@pytest.mark.parametrize("T,k,N", [(500, 6, 4096), (7, 3, 10), (64, 1, 256)])
def test_combine_matches_oracle_and_repeats(B, T, k, N):
    rng = np.random.default_rng(T)
    y = rng.standard_normal((T * k, N)).astype(np.float32)
    s2r = rng.permutation(T * k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    dy, ds, dw = B.to_device(y, DEV), B.to_device(s2r, DEV), B.to_device(w, DEV)
    out = B.combine(dy, ds, dw)
    ref, mag = oracle.combine(y.astype(np.float64), s2r, w)
    _tol_check(out.cpu().numpy(), ref, mag, rel=1e-6, what="combine")
    assert torch.equal(out, B.combine(dy, ds, dw))
    if k == 1:
        np.testing.assert_array_equal(B.combine(dy, ds, B.to_device(np.ones((T, 1), np.float32), DEV))
                                      .cpu().numpy(), y[s2r])


def test_bad_id_leaves_slot_out_and_combine_skips_it(B):
    # An id out of range: MOE_ERR_DATA, slot_to_row = -1 for that slot, and the
    # combine adds nothing for it (it never reads y outside its T*k rows).
    T, k, E, N = 40, 3, 8, 64
    ids = inputs.route_uniform(21, T, E, k)
    bad = 7 * k + 1
    ids.reshape(-1)[bad] = E + 5
    ws = B.make_workspace(T, k, E, DEV)
    gs, off, ss, s2r, _ = B.route_sort(B.to_device(ids, DEV), E, workspace=ws)
    assert B.read_status(ws) == B.MOE_ERR_DATA
    s2r_h = s2r.cpu().numpy()
    assert s2r_h[bad] == -1
    assert int(off[E]) == T * k - 1
    good = np.delete(np.arange(T * k), bad)
    assert sorted(s2r_h[good].tolist()) == list(range(T * k - 1))
    rng = np.random.default_rng(3)
    y = rng.standard_normal((T * k, N)).astype(np.float32)
    w = rng.random((T, k)).astype(np.float32)
    out = B.combine(B.to_device(y, DEV), s2r, B.to_device(w, DEV)).cpu().numpy()
    # Reference: the same sum with the bad slot's weight set to zero.
    s2r_ref, w_ref = s2r_h.copy(), w.copy()
    s2r_ref[bad] = 0
    w_ref.reshape(-1)[bad] = 0.0
    ref, mag = oracle.combine(y.astype(np.float64), s2r_ref, w_ref)
    _tol_check(out, ref, mag, rel=1e-6, what="combine with a skipped slot")


# --------------------------------------------------------------------- layer

def test_layer_forward_stagewise(B):
    c = inputs.layer_case(seed=1, T=96, E=16, hidden=512, inter=256, k=4)
    T, k, E, H, I = c["T"], c["k"], c["E"], c["hidden"], c["inter"]
    bufs = B.LayerBuffers(T, k, E, H, I, DEV)
    out = B.layer_forward(B.bf16_from_bits(c["x"], DEV), B.to_device(c["ids"], DEV),
                          B.to_device(c["topk_w"], DEV), B.to_device(c["w13_codes"], DEV),
                          B.to_device(c["w13_scales"], DEV), B.to_device(c["w2_codes"], DEV),
                          B.to_device(c["w2_scales"], DEV), bufs)
    assert B.last_launch_count() == 8   # route sort 3, w13 2 (band classes), w2 2, combine 1
    assert B.read_status(bufs.workspace) == B.MOE_OK
    gs, off, ss, s2r = oracle.route_sort(c["ids"], E)
    np.testing.assert_array_equal(bufs.slot_to_row.cpu().numpy(), s2r)
    xs = oracle.gather(c["x"], ss, k)
    np.testing.assert_array_equal(k8_deinterleave(B.bits_from_bf16(bufs.x_sorted)), xs)
    # w13 with SwiGLU in its epilogue: h against the oracle's SwiGLU of the
    # oracle's w13 sums (SwiGLU-of-GEMM bound), and bit-identical to the
    # unfused GEMM followed by the SwiGLU kernel.
    y13, m13 = oracle.grouped_gemm(xs, c["w13_codes"], c["w13_scales"], gs)
    h_nat = k8_deinterleave(B.bits_from_bf16(bufs.h))
    check_swiglu_from_gemm(h_nat, y13, m13, oracle.swiglu(y13), what="fused w13 + SwiGLU")
    y13_gpu = B.grouped_gemm(bufs.x_sorted, B.to_device(c["w13_codes"], DEV),
                             B.to_device(c["w13_scales"], DEV), bufs.group_sizes,
                             act_layout=B.MOE_ACT_K8_INTERLEAVED)
    _tol_check(y13_gpu.cpu().numpy(), y13, m13, what="w13")
    np.testing.assert_array_equal(B.bits_from_bf16(bufs.h),
                                  B.bits_from_bf16(B.swiglu(y13_gpu, layout=B.MOE_ACT_K8_INTERLEAVED)))
    y2, m2 = oracle.grouped_gemm(h_nat, c["w2_codes"], c["w2_scales"], gs)
    _tol_check(bufs.y2.cpu().numpy(), y2, m2, what="w2")
    o, mo = oracle.combine(bufs.y2.cpu().numpy().astype(np.float64), s2r, c["topk_w"])
    _tol_check(out.cpu().numpy(), o, mo, rel=1e-6, what="combine")


# ------------------------------------------------------- failure detection

def test_bounded_wait_times_out_and_context_survives(B):
    ws = B.make_workspace(0, 1, 1, DEV)
    B.debug_bounded_wait(2_000_000, ws)          # 2 ms on a barrier nothing completes
    assert B.read_status(ws) == B.MOE_ERR_TIMEOUT
    act, codes, scales, gs = _explicit([10, 0, 3], 128, 128)
    out = _gemm_gpu(B, act, codes, scales, gs)
    ref, mag = oracle.grouped_gemm(act, codes, scales, gs)
    _tol_check(out, ref, mag, what="after timeout")
