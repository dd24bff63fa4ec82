"""GPU parity of the grouped GEMM with one E8M0 scale per 512 k
(moe_mxfp4_grouped_gemm_block), against the fp64 oracle with the same scale
block, in every mode: split (bands <= 32 rows), single (<= 128) and wide
(> 128, K8 activations).  Bar: |gpu - oracle| <= 1e-5 * sum|a w| + 1e-6.
Block 32 through the same entry point equals moe_mxfp4_grouped_gemm bit for bit.
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


def k8_interleave(a):
    a = np.ascontiguousarray(a)
    K = a.shape[-1]
    return a.reshape(*a.shape[:-1], K // 8, 2, 4).swapaxes(-1, -2).reshape(a.shape)


def _case(gs, K, N, seed=0):
    gs = np.asarray(gs, np.int32)
    act = inputs.normal_bf16(seed, 21, (int(gs.sum()), K))
    codes, _ = inputs.mxfp4_weights(seed, 22, len(gs), N, K)
    scales = inputs.e8m0_scales(seed, (len(gs), N, K // 512), 117, 125)
    return act, codes, scales, gs


def _run(B, act, codes, scales, gs, block, k8, out_dtype=torch.float32):
    ws = B.make_workspace(0, 1, 1, DEV)
    a = k8_interleave(act) if k8 else act
    out = B.grouped_gemm_block(B.bf16_from_bits(a, DEV), B.to_device(codes, DEV),
                               B.to_device(scales, DEV), B.to_device(gs, DEV), block,
                               out_dtype=out_dtype, workspace=ws,
                               act_layout=B.MOE_ACT_K8_INTERLEAVED if k8 else B.MOE_ACT_ROW_MAJOR)
    st = B.read_status(ws)
    assert st == B.MOE_OK, B.status_string(st)
    return out


CASES = {
    "split": ([3, 0, 16, 30, 1], 1024, 256),
    "single": ([100, 0, 40, 128], 512, 384),
    "wide": ([300, 129, 0, 17], 1024, 256),
    "mixed_classes": ([1, 200, 0, 64, 20], 2048, 200),
    "layer_k": ([150, 90], 4096, 128),
}


@pytest.mark.parametrize("k8", [False, True], ids=["row_major", "k8"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_block512_matches_oracle(B, name, k8):
    act, codes, scales, gs = _case(*CASES[name])
    out = _run(B, act, codes, scales, gs, 512, k8).cpu().numpy()
    ref, mag = oracle.grouped_gemm_block(act, codes, scales, gs, 512)
    diff = np.abs(out.astype(np.float64) - ref)
    bound = 1e-5 * mag + 1e-6
    assert np.all(diff <= bound), f"{name}: worst ratio {float(np.max(diff / bound)):.3g}"


def test_block512_one_hot_exposes_scale_blocks(B):
    # Identity-like activations: out[row, n] = w[n, k(row)] exactly, for k on
    # both sides of every 512 boundary.
    rng = np.random.default_rng(23)
    K, N = 2048, 128
    codes = rng.integers(0, 256, (1, N, K // 2), dtype=np.uint8)
    scales = rng.integers(110, 140, (1, N, K // 512), dtype=np.uint8)
    kk = np.array([0, 1, 511, 512, 513, 1023, 1024, 1535, 1536, 2047])
    one = inputs.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    act = np.zeros((kk.size, K), np.uint16)
    act[np.arange(kk.size), kk] = one
    out = _run(B, act, codes, scales, np.array([kk.size], np.int32), 512, False).cpu().numpy()
    ref, _ = oracle.grouped_gemm_block(act, codes, scales, np.array([kk.size], np.int32), 512)
    np.testing.assert_array_equal(out, ref)


def test_block32_entry_equals_plain_gemm(B):
    act, codes, _, gs = _case([5, 140, 0, 40], 1024, 256, seed=2)
    scales32 = inputs.e8m0_scales(2, (4, 256, 32), 117, 125)
    plain = B.grouped_gemm(B.bf16_from_bits(act, DEV), B.to_device(codes, DEV),
                           B.to_device(scales32, DEV), B.to_device(gs, DEV))
    viab = _run(B, act, codes, scales32, gs, 32, False)
    assert torch.equal(plain, viab)


def test_block512_flags_out_of_range_scale(B):
    act, codes, scales, gs = _case([20, 3], 1024, 128, seed=4)
    scales[1, 9, 1] = 255
    ws = B.make_workspace(0, 1, 1, DEV)
    B.grouped_gemm_block(B.bf16_from_bits(act, DEV), B.to_device(codes, DEV), B.to_device(scales, DEV),
                         B.to_device(gs, DEV), 512, workspace=ws)
    assert B.read_status(ws) == B.MOE_ERR_DATA
