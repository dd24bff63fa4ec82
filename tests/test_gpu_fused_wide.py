"""GPU parity of the wide mode (256-token work items, taken when a band is over
128 rows and the activations are K8-interleaved) and of the w13 grouped GEMM
with SwiGLU in its epilogue (moe_mxfp4_grouped_gemm_swiglu).

Bars: GEMM f32 outputs within 1e-5 * sum|a w| + 1e-6 of the fp64 oracle; the
fused h bit-identical to the standalone SwiGLU kernel applied to the unfused
GEMM's f32 output (same MMA order, same f32 SwiGLU arithmetic), and within the
SwiGLU-of-GEMM bound (tests/parity_bounds.py) of the oracle's SwiGLU of the
oracle's gate/up sums.
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


def k8_interleave(a):
    a = np.ascontiguousarray(a)
    K = a.shape[-1]
    return a.reshape(*a.shape[:-1], K // 8, 2, 4).swapaxes(-1, -2).reshape(a.shape)


def k8_deinterleave(a):
    a = np.ascontiguousarray(a)
    K = a.shape[-1]
    return a.reshape(*a.shape[:-1], K // 8, 4, 2).swapaxes(-1, -2).reshape(a.shape)


def _tol_check(gpu, ref, mag, rel=1e-5, abs_=1e-6, what=""):
    diff = np.abs(np.asarray(gpu, np.float64) - ref)
    bound = rel * mag + abs_
    bad = ~(diff <= bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {diff.size} outside tolerance; "
                           f"worst ratio {float(np.max(diff / bound)):.3g}")


def _explicit(gs, K, N, seed=0, exp=(-9, -3)):
    gs = np.asarray(gs, np.int32)
    act = inputs.normal_bf16(seed, 11, (int(gs.sum()), K))
    codes, scales = inputs.mxfp4_weights(seed, 12, len(gs), N, K, exp)
    return act, codes, scales, gs


class Dev:
    """Device copies of one case."""

    def __init__(self, B, act, codes, scales, gs, k8):
        self.B = B
        self.act = B.bf16_from_bits(k8_interleave(act) if k8 else act, DEV)
        self.codes, self.scales = B.to_device(codes, DEV), B.to_device(scales, DEV)
        self.gs = B.to_device(np.asarray(gs, np.int32), DEV)
        self.lay = B.MOE_ACT_K8_INTERLEAVED if k8 else B.MOE_ACT_ROW_MAJOR

    def gemm(self):
        B = self.B
        ws = B.make_workspace(0, 1, 1, DEV)
        out = B.grouped_gemm(self.act, self.codes, self.scales, self.gs, workspace=ws,
                             act_layout=self.lay)
        st = B.read_status(ws)
        assert st == B.MOE_OK, B.status_string(st)
        return out

    def fused(self, h_k8):
        B = self.B
        ws = B.make_workspace(0, 1, 1, DEV)
        h = B.grouped_gemm_swiglu(self.act, self.codes, self.scales, self.gs, workspace=ws,
                                  act_layout=self.lay,
                                  h_layout=B.MOE_ACT_K8_INTERLEAVED if h_k8 else B.MOE_ACT_ROW_MAJOR)
        st = B.read_status(ws)
        assert st == B.MOE_OK, B.status_string(st)
        return h


# ------------------------------------------------------------------ wide mode

WIDE_CASES = {
    # band sizes around the 128 / 256 token boundaries, empty and tiny bands
    "bands_129_256_257": lambda: _explicit([129, 0, 256, 257, 1], 512, 256),
    "band_over_1000": lambda: _explicit([1100, 3, 0, 200], 256, 128),
    "mixed_with_small": lambda: _explicit([0, 1, 300, 129, 17, 256, 257, 64, 5], 512, 384),
    # K tails: a partial code stage (K = 288, nine scale bytes a row), one
    # code stage per item (K = 96, 256: the converter pairs alternate items)
    "k_tail_288": lambda: _explicit([300, 40, 140], 288, 200),
    "k_96": lambda: _explicit([150, 7], 96, 136),
    "k_256_many_items": lambda: _explicit([300] * 8, 256, 4096),
    # 192 items over 152 CTAs (one or two each), N = 4096 as in the layer
    "two_items_per_cta": lambda: _explicit([140, 260, 131, 500, 180, 129], 1024, 4096),
    # scale tiles by TMA (K % 512 == 0) with a partial 128-row tile
    "scales_tma_partial_tile": lambda: _explicit([200, 0, 333], 1024, 200),
}


@pytest.mark.parametrize("name", sorted(WIDE_CASES))
def test_wide_mode_matches_oracle(B, name):
    act, codes, scales, gs = WIDE_CASES[name]()
    assert gs.max() > 128
    out = Dev(B, act, codes, scales, gs, k8=True).gemm().cpu().numpy()
    ref, mag = oracle.grouped_gemm(act, codes, scales, gs)
    _tol_check(out, ref, mag, what=name)


def test_wide_mode_identity_activations_expose_decoded_weights(B):
    # Two experts of 256 and 200 rows, K = 512: every act row is one-hot, so
    # out[row, n] = w_e[n, k(row)] exactly; checks the wide mode's token and
    # K placement bit for bit.
    rng = np.random.default_rng(11)
    K, N = 512, 256
    gs = np.array([256, 200], np.int32)
    codes = rng.integers(0, 256, (2, N, K // 2), dtype=np.uint8)
    scales = rng.integers(2, 253, (2, N, K // 32), dtype=np.uint8)
    one = inputs.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    act = np.zeros((456, K), np.uint16)
    kk = np.concatenate([np.arange(256), 300 + np.arange(200)])
    act[np.arange(456), kk] = one
    out = Dev(B, act, codes, scales, gs, k8=True).gemm().cpu().numpy()
    for e, (r0, r1) in enumerate([(0, 256), (256, 456)]):
        dec = inputs.bf16_bits_to_f32(oracle.decode_expert_bf16(codes, scales, e))
        np.testing.assert_array_equal(out[r0:r1], dec[:, kk[r0:r1]].T)


def test_wide_mode_repeatable(B):
    act, codes, scales, gs = WIDE_CASES["mixed_with_small"]()
    d = Dev(B, act, codes, scales, gs, k8=True)
    assert torch.equal(d.gemm(), d.gemm())


# ----------------------------------------------------------- fused SwiGLU

FUSED_CASES = {
    # (bands, K, I): the mode follows the widest band (<= 16 narrow split,
    # <= 32 split, <= 128 single, > 128 wide with K8 activations)
    "narrow_split": ([3, 0, 16, 9], 512, 128),
    "split": ([30, 1, 0, 17], 256, 192),
    "single": ([100, 0, 33, 128], 512, 256),
    "wide": ([300, 129, 0, 40], 512, 256),
    "wide_partial_tiles": ([260, 7], 288, 96),
    "single_partial_tile": ([70, 50], 256, 160),
    "split_partial_tile": ([5, 20], 1024, 80),
    "layer_like": ([190, 200, 0, 180, 230], 1024, 2048),
}


def _fused_case(name, seed=3):
    gs, K, I = FUSED_CASES[name]
    return _explicit(gs, K, 2 * I, seed=seed)


@pytest.mark.parametrize("h_k8", [False, True], ids=["h_rowmajor", "h_k8"])
@pytest.mark.parametrize("act_k8", [False, True], ids=["act_rowmajor", "act_k8"])
@pytest.mark.parametrize("name", sorted(FUSED_CASES))
def test_fused_swiglu_equals_gemm_then_swiglu(B, name, act_k8, h_k8):
    act, codes, scales, gs = _fused_case(name)
    d = Dev(B, act, codes, scales, gs, k8=act_k8)
    y13 = d.gemm()
    want = B.bits_from_bf16(B.swiglu(y13, layout=B.MOE_ACT_K8_INTERLEAVED if h_k8
                                     else B.MOE_ACT_ROW_MAJOR))
    got = B.bits_from_bf16(d.fused(h_k8))
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("name", ["split", "single", "wide", "wide_partial_tiles"])
def test_fused_swiglu_within_bound_of_oracle(B, name):
    act, codes, scales, gs = _fused_case(name, seed=5)
    d = Dev(B, act, codes, scales, gs, k8=True)
    h = k8_deinterleave(B.bits_from_bf16(d.fused(True)))
    y13, mag = oracle.grouped_gemm(act, codes, scales, gs)
    check_swiglu_from_gemm(h, y13, mag, oracle.swiglu(y13), what=name)


def test_fused_swiglu_flags_bad_scale_and_ignores_rows_beyond_i(B):
    # I = 80: the second 64-column tile of expert 0 holds 16 valid gate/up row
    # pairs; its other three 16-row groups lie past I and are zero-filled by
    # the tile load.  Expert 1 is empty and its scale bytes are out of range:
    # never read, no error.
    act, codes, scales, gs = _explicit([20, 0], 512, 160)
    scales[1] = 255
    d = Dev(B, act, codes, scales, gs, k8=False)
    d.fused(False)
    # One out-of-range byte in an up row of expert 0 is an error.
    scales[0, 80 + 5, 3] = 255
    d = Dev(B, act, codes, scales, gs, k8=False)
    ws = B.make_workspace(0, 1, 1, DEV)
    B.grouped_gemm_swiglu(d.act, d.codes, d.scales, d.gs, workspace=ws)
    assert B.read_status(ws) == B.MOE_ERR_DATA


def test_fused_swiglu_rejects_bad_arguments(B):
    act, codes, scales, gs = _explicit([4], 256, 2 * 24)
    d = Dev(B, act, codes, scales, gs, k8=False)
    with pytest.raises(B.MoeError):       # I % 16 != 0 (I = 24)
        B.grouped_gemm_swiglu(d.act, d.codes, d.scales, d.gs)


@pytest.mark.parametrize("bands,K,k8", [
    (np.full(48, 100, np.int32), 768, False),    # single mode, scale bytes by load (K % 512 != 0)
    (np.full(48, 60, np.int32), 512, False),     # single mode, bands <= 64 rows
    (np.full(40, 200, np.int32), 768, True),     # wide mode, scale bytes by load
], ids=["single_ldg_scales", "single_narrow_act", "wide_ldg_scales"])
def test_repeated_launches_are_bitwise_equal(B, bands, K, k8):
    # The converter pairs take alternate code stages; the ring depth must be
    # even so that a pair never waits on a slot last filled for the other pair
    # (whose copy may still be in flight).  Forty launches of shapes whose
    # depth would otherwise be odd must agree bit for bit, and the first must
    # match the oracle on sampled elements.
    act, codes, scales, gs = _explicit(bands, K, 4096, seed=7)
    d = Dev(B, act, codes, scales, gs, k8=k8)
    first = d.gemm()
    for _ in range(40):
        assert torch.equal(d.gemm(), first)
    rng = np.random.default_rng(1)
    r = rng.integers(0, act.shape[0], 4000)
    c = rng.integers(0, 4096, 4000)
    ref, mag = oracle.grouped_gemm_sampled(act, codes, scales, gs, r, c)
    _tol_check(first.cpu().numpy()[r, c], ref, mag, what="repeated launches")


@pytest.mark.parametrize("fused", [False, True], ids=["gemm", "fused_swiglu"])
def test_many_ctas_sharing_weight_tiles_are_bitwise_repeatable(B, fused):
    # One band of 12 full 256-token chunks first, so every CTA's first work
    # item is a full wide item and up to five CTAs read the same weight tile
    # at once: its code-ring refills then hit L2 and land within a few hundred
    # cycles of the slot's release.  The converters' shared-memory reads of a
    # slot must be ordered before that TMA write (a proxy fence); without it,
    # on the full-size Zipf prefill, about one launch in a hundred had a few
    # weight rows of one CTA's first item decoded wrongly.  150 launches must
    # agree bit for bit, and the
    # first must match the oracle on sampled elements.
    act, codes, scales, gs = _explicit([3072, 40, 0, 300], 4096, 4096, seed=9)
    d = Dev(B, act, codes, scales, gs, k8=True)
    run = (lambda: d.fused(True)) if fused else d.gemm
    first = run().clone()
    diffs = [int((run() != first).sum()) for _ in range(150)]
    assert not any(diffs), f"launches differing from the first: {[i for i, n in enumerate(diffs) if n]}"
    if not fused:
        rng = np.random.default_rng(2)
        r = rng.integers(0, act.shape[0], 4000)
        c = rng.integers(0, 4096, 4000)
        ref, mag = oracle.grouped_gemm_sampled(act, codes, scales, gs, r, c)
        _tol_check(first.cpu().numpy()[r, c], ref, mag, what="shared weight tiles")


# ------------------------------------------------------------- CTA pairs

PAIR_CASES = {
    # (bands, K, N, fused): even numbers of column tiles (pairs possible)
    "bands_129_256_257": ([129, 0, 256, 257, 1], 512, 256, False),
    "band_over_1000": ([1100, 3, 0, 200], 256, 512, False),
    "k_tail_288": ([300, 40, 140], 288, 256, False),
    "k_96": ([150, 7, 64], 96, 256, False),
    "many_items": ([140, 260, 131, 500, 180, 129, 33, 48], 1024, 4096, False),
    "scales_by_load": ([200, 0, 333], 768, 512, False),
    "fused_wide": ([300, 129, 0, 40], 512, 2 * 256, True),
    "fused_layer_like": ([190, 200, 0, 180, 230, 35], 1024, 2 * 2048, True),
    "fused_partial_tiles": ([260, 7, 90], 288, 2 * 224, True),
}


@pytest.fixture
def pairing(B):
    yield B
    B.set_gemm_pairing(B.MOE_PAIRING_AUTO)


@pytest.mark.parametrize("name", sorted(PAIR_CASES))
def test_cta_pairs_equal_single_ctas_and_match_oracle(pairing, name):
    # The CTA-pair kernel (M = 256 MMAs over two SMs, each SM loading half of
    # every activation tile) must give the single-CTA kernel's results bit for
    # bit (same products, same accumulation order), and the oracle's.
    B = pairing
    gs, K, N, fused = PAIR_CASES[name]
    act, codes, scales, gs = _explicit(gs, K, N, seed=13)
    d = Dev(B, act, codes, scales, gs, k8=True)
    run = (lambda: d.fused(True)) if fused else d.gemm
    B.set_gemm_pairing(B.MOE_PAIRING_OFF)
    single = run()
    B.set_gemm_pairing(B.MOE_PAIRING_ON)
    paired = run()
    assert torch.equal(paired, single)
    if fused:
        h = k8_deinterleave(B.bits_from_bf16(paired))
        y13, mag = oracle.grouped_gemm(act, codes, scales, gs)
        check_swiglu_from_gemm(h, y13, mag, oracle.swiglu(y13), what=name)
    else:
        ref, mag = oracle.grouped_gemm(act, codes, scales, gs)
        _tol_check(paired.cpu().numpy(), ref, mag, what=name)


def test_cta_pairs_repeatable_with_many_ctas_per_weight_tile(pairing):
    # As test_many_ctas_sharing_weight_tiles_are_bitwise_repeatable, in pairs.
    B = pairing
    act, codes, scales, gs = _explicit([3072, 40, 0, 300], 4096, 4096, seed=9)
    d = Dev(B, act, codes, scales, gs, k8=True)
    B.set_gemm_pairing(B.MOE_PAIRING_ON)
    first = d.gemm().clone()
    diffs = [int((d.gemm() != first).sum()) for _ in range(60)]
    assert not any(diffs), f"launches differing from the first: {[i for i, n in enumerate(diffs) if n]}"
    B.set_gemm_pairing(B.MOE_PAIRING_OFF)
    assert torch.equal(d.gemm(), first)


def test_pairing_mode_rejects_unknown_values(B):
    with pytest.raises(B.MoeError):
        B.set_gemm_pairing(3)
