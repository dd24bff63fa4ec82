"""GPU parity of the lossless MXFP4 -> NVFP4 scale cast ("DeepSeek-V4-Flash-0731-
NVFP4", "The lossless weight cast"), called through the C ABI, against the CPU
oracle on the same seeded scales.

Bar: bit-exact E4M3 bytes, per-tensor f32 scales and out-of-range counts (all
integer or exactly representable results).  Independently of the oracle, every
in-range block must dequantize to exactly its MXFP4 scale:
E4M3 value x weight_scale_2 == 2^(s - 127).
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


ONE_PASS_MAX = 8 * 64 * 1024     # bytes of one expert's scales that one cluster holds


def _expected_launches(shape, src_ptr=0, dst_ptr=0):
    """One cluster kernel when an expert's scales are a multiple of 16 bytes, at
    most 512 KiB, and both buffers start on 16-byte boundaries; else two passes."""
    per = shape[1] * shape[2]
    one = per % 16 == 0 and per <= ONE_PASS_MAX and src_ptr % 16 == 0 and dst_ptr % 16 == 0
    return 1 if one else 2


def _cast(B, scales_np):
    s = torch.from_numpy(np.ascontiguousarray(scales_np)).to(DEV)
    ws = torch.empty(int(B.load().moe_nvfp4_cast_workspace_bytes(s.shape[0])), dtype=torch.uint8,
                     device=DEV)
    B.clear_status(ws)
    e4m3, ws2, oob = B.mxfp4_to_nvfp4(s, workspace=ws)
    st = B.read_status(ws)
    assert B.last_launch_count() == _expected_launches(s.shape)
    return e4m3.cpu().numpy(), ws2.cpu().numpy(), oob.cpu().numpy(), st


def _check_against_oracle(B, scales):
    e4m3, ws2, oob, st = _cast(B, scales)
    assert st == B.MOE_OK
    o_e4m3, o_ws2, o_oob = oracle.mxfp4_to_nvfp4(scales)
    np.testing.assert_array_equal(e4m3, o_e4m3)
    # weight_scale_2 is a power of two >= 2^-135, exact in f32 (subnormal below 2^-126).
    np.testing.assert_array_equal(ws2.astype(np.float64), o_ws2)
    np.testing.assert_array_equal(oob, o_oob)
    return e4m3, ws2, oob


def _dequant_exact(scales, e4m3, ws2):
    """In-range blocks: E4M3 value x weight_scale_2 == 2^(s - 127), computed from
    the GPU's bytes with torch's float8_e4m3fn decoding (not the oracle)."""
    E = scales.shape[0]
    vals = torch.from_numpy(e4m3.reshape(-1)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vals = vals.reshape(e4m3.shape)
    want = np.ldexp(1.0, scales.astype(np.int64) - 127)
    got0 = vals[..., 0::2] * ws2.astype(np.float64).reshape(E, 1, 1)
    got1 = vals[..., 1::2] * ws2.astype(np.float64).reshape(E, 1, 1)
    ok = e4m3[..., 0::2] != 0
    np.testing.assert_array_equal(got0[ok], want[ok])
    np.testing.assert_array_equal(got1[ok], want[ok])
    np.testing.assert_array_equal(e4m3[..., 0::2], e4m3[..., 1::2])
    return int((~ok).sum())


CASES = {
    # The workload exponent range [-10, -2]: every block in range.
    "typical": ((8, 64, 8), 117, 125),
    # Every byte but the NaN: most blocks out of range.
    "full_range": ((4, 96, 16), 0, 254),
    # 19 binades: byte m - 17 is the last exact one (E4M3 2^-9), m - 18 is out.
    "edge_19": ((16, 32, 4), 99, 117),
    # Ragged: expert tensors of 37 * 3 = 111 bytes (odd strides, unaligned bases).
    "ragged": ((5, 37, 3), 90, 140),
    # One expert split into 131 chunks; the last one ends in a 6-byte tail.
    "one_expert_wide": ((1, 4099, 130), 110, 127),
    # Many experts, one chunk each (one pass: clusters of one CTA).
    "many_experts": ((1024, 8, 2), 60, 130),
    # One pass with 2 CTAs per cluster, the second one partly filled.
    "cluster_2": ((3, 1000, 100), 100, 127),
    # One pass with 5 CTAs per cluster.
    "cluster_5": ((2, 2560, 128), 110, 125),
    # One pass with 8 CTAs per cluster, the last one partly filled; fewer experts
    # than resident clusters.
    "cluster_8_ragged": ((3, 4000, 128), 100, 127),
    # The w2 scale tensor of the workloads: clusters of 4, many experts per cluster.
    "w2_shape": ((256, 4096, 64), 117, 125),
    # Aligned but over 512 KiB per expert: two passes, 16-byte vector path.
    "two_pass_aligned": ((2, 4096, 160), 110, 127),
    # The same over every byte but the NaN: two passes with blocks out of range.
    "two_pass_full_range": ((1, 8192, 80), 0, 254),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_cast_matches_oracle(B, name):
    shape, lo, hi = CASES[name]
    scales = inputs.e8m0_scales(0, shape, lo, hi)
    e4m3, ws2, oob = _check_against_oracle(B, scales)
    zeros = _dequant_exact(scales, e4m3, ws2)
    assert zeros == int(oob.sum())
    if name == "typical":
        assert int(oob.sum()) == 0


def test_cast_special_experts(B):
    """All-zero scales (per-tensor scale 2^-135, an f32 subnormal), the largest
    finite byte 254 (2^119), exactly 17 binades (the lowest still exact, as the
    E4M3 subnormal 2^-9) and 18 binades (one block written as 0)."""
    N, nb = 16, 4
    scales = np.full((4, N, nb), 200, np.uint8)
    scales[0] = 0
    scales[1] = 254
    scales[1, 3, 2] = 254 - 17
    scales[2] = 150
    scales[2, 0, 0] = 150 - 17
    scales[3] = 150
    scales[3, 5, 1] = 150 - 18
    e4m3, ws2, oob = _check_against_oracle(B, scales)
    assert ws2[0] == np.float32(2.0 ** -135) and ws2[0] > 0
    assert ws2[1] == np.float32(2.0 ** 119)
    assert e4m3[0].min() == e4m3[0].max() == 0x78          # 2^8 for every block at the max
    assert e4m3[1, 3, 4] == e4m3[1, 3, 5] == 0x01           # 2^-9
    assert e4m3[2, 0, 0] == 0x01
    assert e4m3[3, 5, 2] == e4m3[3, 5, 3] == 0
    assert oob.tolist() == [0, 0, 0, 1]
    _dequant_exact(scales, e4m3, ws2)


def test_cast_w13_full_size_and_repeatable(B):
    """The w13 scale tensor of the workloads (256 experts x 4096 rows x 128
    blocks, 128 MiB), bit-exact against the oracle, and twice in a row bitwise
    equal."""
    scales = inputs.e8m0_scales(0, (256, 4096, 128), 117, 125)
    e4m3, ws2, oob = _check_against_oracle(B, scales)
    assert int(oob.sum()) == 0
    e4m3b, ws2b, oobb, st = _cast(B, scales)
    assert st == B.MOE_OK
    np.testing.assert_array_equal(e4m3, e4m3b)
    np.testing.assert_array_equal(ws2, ws2b)
    np.testing.assert_array_equal(oob, oobb)


@pytest.mark.parametrize("src_off,dst_off", [(8, 0), (3, 0), (0, 5), (7, 9)])
def test_cast_unaligned_buffers(B, src_off, dst_off):
    """Scale input and E4M3 output at byte offsets away from 16-byte boundaries:
    (8, 0) takes an 8-byte single-byte head before the vector path; in the
    other cases the output never lines up and every byte takes the single-byte
    path."""
    shape = (6, 53, 5)
    scales = inputs.e8m0_scales(2, shape, 95, 125)
    n = scales.size
    sbuf = torch.zeros(n + 16, dtype=torch.uint8, device=DEV)
    sbuf[src_off:src_off + n] = torch.from_numpy(scales.reshape(-1)).to(DEV)
    obuf = torch.full((2 * n + 16,), 0xEE, dtype=torch.uint8, device=DEV)
    e4m3 = obuf[dst_off:dst_off + 2 * n].view(shape[0], shape[1], 2 * shape[2])
    ws2 = torch.empty(shape[0], dtype=torch.float32, device=DEV)
    oob = torch.empty(shape[0], dtype=torch.int64, device=DEV)
    ws = torch.empty(int(B.load().moe_nvfp4_cast_workspace_bytes(shape[0])), dtype=torch.uint8,
                     device=DEV)
    B.clear_status(ws)
    B.mxfp4_to_nvfp4(sbuf[src_off:src_off + n].view(shape), out=(e4m3, ws2, oob), workspace=ws)
    assert B.read_status(ws) == B.MOE_OK
    assert B.last_launch_count() == 2
    o_e4m3, o_ws2, o_oob = oracle.mxfp4_to_nvfp4(scales)
    np.testing.assert_array_equal(e4m3.cpu().numpy(), o_e4m3)
    np.testing.assert_array_equal(ws2.cpu().numpy().astype(np.float64), o_ws2)
    np.testing.assert_array_equal(oob.cpu().numpy(), o_oob)
    # Nothing written outside the output view.
    ob = obuf.cpu().numpy()
    assert (ob[:dst_off] == 0xEE).all() and (ob[dst_off + 2 * n:] == 0xEE).all()


def test_cast_flags_nan_scale(B):
    scales = inputs.e8m0_scales(1, (3, 40, 8), 100, 130)
    scales[1, 17, 5] = 255
    with pytest.raises(ValueError):
        oracle.mxfp4_to_nvfp4(scales)
    _, _, _, st = _cast(B, scales)
    assert st == B.MOE_ERR_DATA


def test_cast_rejects_bad_arguments(B):
    lib = B.load()
    s = torch.zeros((2, 4, 2), dtype=torch.uint8, device=DEV)
    o = torch.zeros((2, 4, 4), dtype=torch.uint8, device=DEV)
    f = torch.zeros(2, dtype=torch.float32, device=DEV)
    c = torch.zeros(2, dtype=torch.int64, device=DEV)
    ws = torch.zeros(int(lib.moe_nvfp4_cast_workspace_bytes(2)), dtype=torch.uint8, device=DEV)
    P = B._ptr
    stream = B._stream()

    def call(E=2, N=4, K=64, wsb=None):
        return lib.moe_mxfp4_to_nvfp4(P(s), E, N, K, P(o), P(f), P(c), P(ws),
                                      ws.numel() if wsb is None else wsb, stream)

    assert call() == B.MOE_OK
    assert call(K=48) == B.MOE_ERR_INVALID_ARG
    assert call(E=0) == B.MOE_ERR_INVALID_ARG
    assert call(N=0) == B.MOE_ERR_INVALID_ARG
    assert call(wsb=256) == B.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
