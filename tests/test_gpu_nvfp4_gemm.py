"""GPU parity of the NVFP4 W4A16 grouped GEMM ("Running DeepSeek V4 Flash on
TPU v6", section 1: the NVFP4 kernel decoding e2m1 weights and per-16 E4M3
scales; "DeepSeek-V4-Flash-0731-NVFP4", "The lossless weight cast": per-16 E4M3
scales under a per-tensor weight_scale_2), called through the C ABI.

Bars: f32 outputs within |gpu - oracle| <= 1e-5 * sum_k |a_k w_k| + 1e-6 of the
fp64 oracle (bf16 outputs: one bf16 ulp more); weights cast losslessly from
MXFP4 give exactly the MXFP4 GEMM's outputs; NaN scales are flagged.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_weight_grouped_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as g
    g.build()
    from fp4_weight_grouped_gb300 import binding
    binding.load()
    return binding


def _tol_check(gpu, ref, mag, extra=None, what=""):
    gpu = np.asarray(gpu, np.float64)
    bound = 1e-5 * mag + 1e-6
    if extra is not None:
        bound = bound + extra
    diff = np.abs(gpu - ref)
    bad = ~(diff <= bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {diff.size} outside tolerance; "
                           f"worst ratio {float(np.max(diff / bound)):.3g}")


def _bf16_ulp(x):
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    return np.ldexp(1.0, (np.maximum(e, -126) - 7).astype(np.int64))


def _k8(a):
    a = np.ascontiguousarray(a)
    K = a.shape[-1]
    return a.reshape(*a.shape[:-1], K // 8, 2, 4).swapaxes(-1, -2).reshape(a.shape)


def _case(gs, K, N, seed=0, lo=0x28, hi=0x48):
    gs = np.asarray(gs, np.int32)
    E = len(gs)
    act = inputs.normal_bf16(seed, 21, (int(gs.sum()), K))
    codes, _ = inputs.mxfp4_weights(seed, 22, E, N, K)
    s16 = inputs.e4m3_scales(seed, (E, N, K // 16), lo, hi, signs=True)
    ws2 = inputs.tensor_scales(seed, E)
    return act, codes, s16, ws2, gs


def _nv_gpu(B, act, codes, s16, ws2, gs, out_dtype=torch.float32, k8=False, s16_dev=None):
    ws = B.make_workspace(0, 1, 1, DEV)
    a = _k8(act) if k8 else act
    out = B.nvfp4_grouped_gemm(B.bf16_from_bits(a, DEV), B.to_device(codes, DEV),
                               B.to_device(s16, DEV) if s16_dev is None else s16_dev,
                               B.to_device(ws2, DEV), B.to_device(gs, DEV), out_dtype=out_dtype,
                               workspace=ws,
                               act_layout=B.MOE_ACT_K8_INTERLEAVED if k8 else B.MOE_ACT_ROW_MAJOR)
    st = B.read_status(ws)
    assert B.last_launch_count() == (2 if act.shape[0] else 0)   # one launch per band class
    return out, st


CASES = {
    # single mode (bands > 32 rows) with every band class; scales by TMA (K % 256 == 0)
    "ragged_bands": ([0, 1, 15, 16, 17, 127, 128, 129, 300, 0, 5], 512, 256),
    # K tails: scales read with loads, the last code stage partly beyond K
    "k_tail_96": ([9, 0, 33], 96, 200),
    "k_tail_160": ([40, 3], 160, 136),
    # split mode (bands <= 32), and narrow split mode (bands <= 16)
    "split_small_bands": ([0, 1, 7, 16, 0, 3, 32, 12, 17, 31], 1024, 384),
    "split_narrow": ([16, 5, 0, 9], 256, 128),
    "split_k_96": ([3, 0, 8], 96, 128),
    "one_expert_long_band": ([700], 256, 128),
}


@pytest.mark.parametrize("k8", [False, True], ids=["row_major", "k8"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_nvfp4_gemm_matches_oracle(B, name, k8):
    act, codes, s16, ws2, gs = _case(*CASES[name])
    out, st = _nv_gpu(B, act, codes, s16, ws2, gs, k8=k8)
    assert st == B.MOE_OK, B.status_string(st)
    ref, mag = oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, gs)
    _tol_check(out.cpu().numpy(), ref, mag, what=name)


def test_nvfp4_gemm_wide_scale_range_and_bf16_output(B):
    # every finite E4M3 magnitude from the smallest subnormal to 448
    act, codes, s16, ws2, gs = _case([5, 0, 130, 17], 384, 256, seed=1, lo=0x01, hi=0x7E)
    out, st = _nv_gpu(B, act, codes, s16, ws2, gs, out_dtype=torch.bfloat16)
    assert st == B.MOE_OK
    ref, mag = oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, gs)
    got = inputs.bf16_bits_to_f32(B.bits_from_bf16(out))
    _tol_check(got, ref, mag, extra=_bf16_ulp(ref), what="bf16 out")


@pytest.mark.parametrize("offset", [1, 8], ids=["byte_aligned", "8_byte_aligned"])
def test_nvfp4_gemm_scales_at_unaligned_address(B, offset):
    act, codes, s16, ws2, gs = _case([40, 3, 9], 512, 128, seed=2)
    buf = torch.zeros(s16.size + 16, dtype=torch.uint8, device=DEV)
    buf[offset:offset + s16.size] = torch.from_numpy(s16.reshape(-1)).to(DEV)
    out, st = _nv_gpu(B, act, codes, s16, ws2, gs, s16_dev=buf[offset:offset + s16.size].view(s16.shape))
    assert st == B.MOE_OK
    ref, mag = oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, gs)
    _tol_check(out.cpu().numpy(), ref, mag, what=f"scales at +{offset}")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("gs,K,N", [([0, 1, 15, 16, 17, 127, 128, 129, 300, 0, 5], 512, 256),
                                    ([0, 1, 7, 16, 0, 3, 32, 12, 17, 31], 1024, 384),
                                    ([9, 0, 33], 96, 200)],
                         ids=["single", "split", "k_tail"])
def test_lossless_cast_then_nvfp4_gemm_equals_mxfp4_gemm(B, gs, K, N, out_dtype):
    """Cast weights dequantize to the MXFP4 values; each NVFP4 weight is the
    MXFP4 weight times an exact power of two that the epilogue undoes, so the
    outputs are bitwise those of the MXFP4 GEMM."""
    gs = np.asarray(gs, np.int32)
    E = len(gs)
    act = inputs.normal_bf16(3, 23, (int(gs.sum()), K))
    codes, scales = inputs.mxfp4_weights(3, 24, E, N, K, (-9, -3))
    a, c, g = B.bf16_from_bits(act, DEV), B.to_device(codes, DEV), B.to_device(gs, DEV)
    ws = B.make_workspace(0, 1, 1, DEV)
    mx = B.grouped_gemm(a, c, B.to_device(scales, DEV), g, out_dtype=out_dtype, workspace=ws)
    e4m3, ws2, oob = B.mxfp4_to_nvfp4(B.to_device(scales, DEV))
    assert int(oob.sum()) == 0
    nv = B.nvfp4_grouped_gemm(a, c, e4m3, ws2, g, out_dtype=out_dtype, workspace=ws)
    assert B.read_status(ws) == B.MOE_OK
    bits = torch.int32 if out_dtype == torch.float32 else torch.int16
    assert torch.equal(mx.view(bits), nv.view(bits))


def test_nvfp4_gemm_flags_nan_scale_and_skips_empty_experts(B):
    act, codes, s16, ws2, gs = _case([7, 0, 20], 256, 128, seed=4)
    s16 = s16.copy()
    s16[1, 3, 2] = 0x7F                 # expert 1 is empty: never read
    out, st = _nv_gpu(B, act, codes, s16, ws2, gs)
    assert st == B.MOE_OK
    s16[2, 100, 5] = 0xFF               # used row of expert 2
    _, st = _nv_gpu(B, act, codes, s16, ws2, gs)
    assert st == B.MOE_ERR_DATA


def test_nvfp4_gemm_repeatable(B):
    act, codes, s16, ws2, gs = _case([0, 1, 7, 16, 0, 3, 32, 12, 17, 31], 1024, 384, seed=5)
    a, _ = _nv_gpu(B, act, codes, s16, ws2, gs)
    b, _ = _nv_gpu(B, act, codes, s16, ws2, gs)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_nvfp4_cta_pairs_equal_single_ctas(B):
    # Bands over 32 rows with an even tile count run in CTA pairs: identical
    # to one CTA per item, bit for bit.
    rng = np.random.default_rng(21)
    gs = np.array([300, 129, 0, 40, 257], np.int32)
    K, N = 512, 512
    act = inputs.normal_bf16(21, 1, (int(gs.sum()), K))
    codes = rng.integers(0, 256, (len(gs), N, K // 2), dtype=np.uint8)
    s16 = rng.integers(0x28, 0x48, (len(gs), N, K // 16), dtype=np.uint8)
    ws2 = np.ldexp(1.0, rng.integers(-6, 3, len(gs))).astype(np.float32)
    k8 = act.reshape(act.shape[0], K // 8, 2, 4).swapaxes(-1, -2).reshape(act.shape)
    d = [B.bf16_from_bits(k8, DEV), B.to_device(codes, DEV), B.to_device(s16, DEV),
         B.to_device(ws2, DEV), B.to_device(gs, DEV)]
    try:
        B.set_gemm_pairing(B.MOE_PAIRING_OFF)
        single = B.nvfp4_grouped_gemm(*d, act_layout=B.MOE_ACT_K8_INTERLEAVED)
        B.set_gemm_pairing(B.MOE_PAIRING_ON)
        paired = B.nvfp4_grouped_gemm(*d, act_layout=B.MOE_ACT_K8_INTERLEAVED)
    finally:
        B.set_gemm_pairing(B.MOE_PAIRING_AUTO)
    assert torch.equal(paired, single)
    ref, mag = oracle.nvfp4_grouped_gemm(act, codes, s16, ws2, gs)
    diff = np.abs(paired.cpu().numpy().astype(np.float64) - ref)
    assert np.all(diff <= 1e-5 * mag + 1e-6), float((diff / (1e-5 * mag + 1e-6)).max())
