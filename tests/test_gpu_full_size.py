"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark times (one persistent CTA per SM).

  decode w13 (T = 64, 384 rows) and decode w2 (T = 256, 1536 rows): every
      output element against the fp64 oracle.
  prefill w13 (T = 4096, 24576 rows, Zipf routing): 16 random elements of
      every (expert, 128-column tile) pair plus the first and last row of
      every band; the full product would take the oracle about a minute.
  layer (T = 8192, 49152 rows, w13 with SwiGLU in its epilogue): route sort
      and gather bit-exact in full; the fused h bit-identical in full to the
      unfused w13 GEMM followed by the SwiGLU kernel, that SwiGLU within 1 bf16
      ulp of the oracle in full, h sampled against the oracle's own w13 sums;
      the w13 and w2 GEMMs sampled as for prefill; combine (fed the GPU's y2)
      compared element by element.

Bars as in test_gpu_parity: GEMM |gpu - oracle| <= 1e-5 * sum|a w| + 1e-6;
SwiGLU within 1 bf16 ulp; combine within 1e-6 * sum|w y| + 1e-6.
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


def _tol_check(gpu, ref, mag, rel=1e-5, abs_=1e-6, what=""):
    gpu = np.asarray(gpu, np.float64)
    bound = rel * mag + abs_
    diff = np.abs(gpu - ref)
    bad = ~(diff <= bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {diff.size} outside tolerance; "
                           f"worst ratio {float(np.max(diff / bound)):.3g}")


def k8_deinterleave(a):
    a = np.ascontiguousarray(a)
    K = a.shape[-1]
    return a.reshape(*a.shape[:-1], K // 8, 4, 2).swapaxes(-1, -2).reshape(a.shape)


def tile_samples(gs, N, per_tile=16, seed=0):
    """(row, col) samples: `per_tile` random elements of every (non-empty
    expert, 128-column tile) pair, plus the first and last row of every band
    at a random column and at column N - 1."""
    rng = np.random.default_rng(seed)
    gs = np.asarray(gs, np.int64)
    off = np.concatenate([[0], np.cumsum(gs)])
    ne = np.nonzero(gs)[0]
    n_tiles = (N + 127) // 128
    e = np.repeat(ne, n_tiles * per_tile)
    tile = np.tile(np.repeat(np.arange(n_tiles), per_tile), ne.size)
    r = off[e] + (rng.random(e.size) * gs[e]).astype(np.int64)
    width = np.minimum(128, N - tile * 128)
    c = tile * 128 + (rng.random(e.size) * width).astype(np.int64)
    edge = np.concatenate([off[ne], off[ne + 1] - 1])
    r = np.concatenate([r, edge, edge])
    c = np.concatenate([c, rng.integers(0, N, edge.size), np.full(edge.size, N - 1)])
    return r.astype(np.int64), c.astype(np.int64)


def test_tile_samples_cover_every_expert_tile_pair():
    gs = np.array([3, 0, 300, 1], np.int32)
    r, c = tile_samples(gs, 520, per_tile=2)
    off = np.concatenate([[0], np.cumsum(gs)])
    e_of_row = np.searchsorted(off, r, side="right") - 1
    pairs = set(zip(e_of_row.tolist(), (c // 128).tolist()))
    assert pairs == {(e, t) for e in (0, 2, 3) for t in range(5)}
    assert r.max() < gs.sum() and c.max() == 519


def _gemm(B, act_bits, codes, scales, gs_dev):
    ws = B.make_workspace(0, 1, 1, DEV)
    out = B.grouped_gemm(B.bf16_from_bits(act_bits, DEV), B.to_device(codes, DEV),
                         B.to_device(scales, DEV), gs_dev, workspace=ws)
    st = B.read_status(ws)
    assert st == B.MOE_OK, B.status_string(st)
    return out.cpu().numpy()


@pytest.mark.parametrize("name", ["decode_w13", "decode_w2"])
def test_decode_gemm_every_element(B, name):
    c = inputs.gemm_case(name)
    gs, *_ = oracle.route_sort(c["ids"], c["E"])
    g_gs = B.route_sort(B.to_device(c["ids"], DEV), c["E"])[0]
    np.testing.assert_array_equal(g_gs.cpu().numpy(), gs)
    out = _gemm(B, c["act"], c["codes"], c["scales"], g_gs)
    ref, mag = oracle.grouped_gemm(c["act"], c["codes"], c["scales"], gs)
    _tol_check(out, ref, mag, what=name)


def test_prefill_gemm_every_tile_sampled(B):
    c = inputs.gemm_case("prefill_w13")
    gs, *_ = oracle.route_sort(c["ids"], c["E"])
    assert int((gs == 0).sum()) == 20 and int(gs.max()) > 1000
    g_gs = B.route_sort(B.to_device(c["ids"], DEV), c["E"])[0]
    np.testing.assert_array_equal(g_gs.cpu().numpy(), gs)
    out = _gemm(B, c["act"], c["codes"], c["scales"], g_gs)
    assert np.isfinite(out).all()
    r, col = tile_samples(gs, c["N"])
    assert r.size >= 100_000
    ref, mag = oracle.grouped_gemm_sampled(c["act"], c["codes"], c["scales"], gs, r, col)
    _tol_check(out[r, col], ref, mag, what="prefill w13")


def test_layer_full_size_stagewise(B):
    c = inputs.layer_case(seed=0)
    T, k, E, H, I = c["T"], c["k"], c["E"], c["hidden"], c["inter"]
    bufs = B.LayerBuffers(T, k, E, H, I, DEV)
    d_w13c, d_w13s = B.to_device(c["w13_codes"], DEV), B.to_device(c["w13_scales"], DEV)
    d_w2c, d_w2s = B.to_device(c["w2_codes"], DEV), B.to_device(c["w2_scales"], DEV)
    out = B.layer_forward(B.bf16_from_bits(c["x"], DEV), B.to_device(c["ids"], DEV),
                          B.to_device(c["topk_w"], DEV), d_w13c, d_w13s, d_w2c, d_w2s, bufs)
    st = B.read_status(bufs.workspace)
    assert st == B.MOE_OK, B.status_string(st)

    # route sort and gather: bit-exact in full
    gs, off, ss, s2r = oracle.route_sort(c["ids"], E)
    np.testing.assert_array_equal(bufs.group_sizes.cpu().numpy(), gs)
    np.testing.assert_array_equal(bufs.group_offsets.cpu().numpy(), off)
    np.testing.assert_array_equal(bufs.sorted_slot.cpu().numpy(), ss)
    np.testing.assert_array_equal(bufs.slot_to_row.cpu().numpy(), s2r)
    xs = oracle.gather(c["x"], ss, k)
    np.testing.assert_array_equal(k8_deinterleave(B.bits_from_bf16(bufs.x_sorted)), xs)

    # w13 with SwiGLU fused: (1) the unfused GEMM, every (expert, column tile)
    # pair sampled against the oracle; (2) the fused h bit-identical, every
    # element, to the SwiGLU kernel applied to that GEMM's f32 output; (3) the
    # SwiGLU kernel within 1 bf16 ulp of the oracle fed the same f32 sums,
    # every element; (4) h sampled against the oracle's SwiGLU of the
    # oracle's own gate/up sums.
    K8 = B.MOE_ACT_K8_INTERLEAVED
    y13_d = B.grouped_gemm(bufs.x_sorted, d_w13c, d_w13s, bufs.group_sizes, act_layout=K8)
    y13 = y13_d.cpu().numpy()
    assert np.isfinite(y13).all()
    r, col = tile_samples(gs, 2 * I, seed=1)
    ref, mag = oracle.grouped_gemm_sampled(xs, c["w13_codes"], c["w13_scales"], gs, r, col)
    _tol_check(y13[r, col], ref, mag, what="layer w13")
    h_unfused = B.swiglu(y13_d, layout=K8)
    np.testing.assert_array_equal(B.bits_from_bf16(bufs.h), B.bits_from_bf16(h_unfused))
    del y13_d, h_unfused
    h_nat = k8_deinterleave(B.bits_from_bf16(bufs.h))
    h_ref = oracle.swiglu(y13)
    del y13
    assert np.abs(h_nat.astype(np.int64) - h_ref.astype(np.int64)).max() <= 1
    del h_ref
    rh, ih = tile_samples(gs, I, per_tile=32, seed=3)
    gu_ref, gu_mag = oracle.grouped_gemm_sampled(
        xs, c["w13_codes"], c["w13_scales"], gs, np.concatenate([rh, rh]), np.concatenate([ih, I + ih]))
    n = rh.size
    y_pair = np.stack([gu_ref[:n], gu_ref[n:]], axis=1)
    m_pair = np.stack([gu_mag[:n], gu_mag[n:]], axis=1)
    check_swiglu_from_gemm(h_nat[rh, ih][:, None], y_pair, m_pair, oracle.swiglu(y_pair),
                           what="layer h (fused) vs oracle")

    # w2: sampled, the oracle fed the GPU's h
    y2 = bufs.y2.cpu().numpy()
    r, col = tile_samples(gs, H, seed=2)
    ref, mag = oracle.grouped_gemm_sampled(h_nat, c["w2_codes"], c["w2_scales"], gs, r, col)
    _tol_check(y2[r, col], ref, mag, what="layer w2")

    # combine: every element, the oracle fed the GPU's y2
    o, mo = oracle.combine(y2, s2r, c["topk_w"])
    _tol_check(out.cpu().numpy(), o, mo, rel=1e-6, what="layer combine")
