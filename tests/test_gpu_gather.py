"""GPU parity of the routing permutations fused into the grouped GEMMs ("Running
DeepSeek V4 Flash on TPU v6", section 1: the activation permutation that the
grouped-matmul timings leave out):

  moe_mxfp4_grouped_gemm_swiglu_gather  sorted row r reads token row
      sorted_slot[r] // k of x_k8 through four-row TMA gathers: h must equal,
      bit for bit, moe_mxfp4_grouped_gemm_swiglu on the gathered copy, in every
      kernel mode (split, narrow split, single, wide) and h layout.
  moe_mxfp4_grouped_gemm_scatter  sorted row r written to row out_row[r]: equal
      bit for bit to moe_mxfp4_grouped_gemm permuted on the host; an entry out
      of range is skipped and flagged.
  moe_combine_slots  y in slot order: equal bit for bit to moe_combine on the
      sorted rows (same FMA chain), bad ids skipped.
  moe_act_interleave_k8  the K8 order, bit-exact.
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


def routing_with_bands(gs, k, seed):
    """topk_ids [T, k] whose expert e receives exactly gs[e] slots (sum(gs) a
    multiple of k), in a random slot order."""
    gs = np.asarray(gs, np.int64)
    ids = np.repeat(np.arange(gs.size, dtype=np.int32), gs)
    np.random.default_rng(seed).shuffle(ids)
    return ids.reshape(-1, k)


class Case:
    def __init__(self, B, gs, k, K, N, seed=0, exp=(-9, -3)):
        self.B = B
        self.ids = routing_with_bands(gs, k, seed)
        self.T, self.k = self.ids.shape
        self.E = len(gs)
        self.x = inputs.normal_bf16(seed, 21, (self.T, K))
        self.codes, self.scales = inputs.mxfp4_weights(seed, 22, self.E, N, K, exp)
        d_ids = B.to_device(self.ids, DEV)
        self.gs, self.off, self.ss, self.s2r = B.route_sort(d_ids, self.E)[:4]
        self.x_k8 = B.bf16_from_bits(k8_interleave(self.x), DEV)
        self.x_sorted = self.x_k8[self.ss.long() // self.k]     # the gathered copy (reference)
        self.d_codes, self.d_scales = B.to_device(self.codes, DEV), B.to_device(self.scales, DEV)

    def ws(self):
        return self.B.make_workspace(0, 1, 1, DEV)


GATHER_CASES = {
    # (bands, k, K, I): the mode follows the widest band of each band class
    "narrow_split": ([3, 0, 16, 9, 4], 4, 512, 128),
    "split": ([30, 1, 0, 17, 32], 5, 256, 192),
    "single": ([100, 0, 33, 128, 7], 4, 512, 256),
    "wide": ([300, 129, 0, 40, 3], 4, 512, 256),
    "wide_partial_tiles": ([260, 7, 33], 3, 288, 96),
    "layer_like": ([190, 200, 0, 180, 230, 16], 6, 1024, 2048),
    "one_big_band": ([3072, 40, 0, 296], 4, 4096, 2048),
}


@pytest.mark.parametrize("h_k8", [False, True], ids=["h_rowmajor", "h_k8"])
@pytest.mark.parametrize("name", sorted(GATHER_CASES))
def test_gather_equals_gemm_on_gathered_rows(B, name, h_k8):
    gs, k, K, I = GATHER_CASES[name]
    c = Case(B, gs, k, K, 2 * I, seed=4)
    lay = B.MOE_ACT_K8_INTERLEAVED if h_k8 else B.MOE_ACT_ROW_MAJOR
    ws1, ws2 = c.ws(), c.ws()
    want = B.grouped_gemm_swiglu(c.x_sorted, c.d_codes, c.d_scales, c.gs, workspace=ws1,
                                 act_layout=B.MOE_ACT_K8_INTERLEAVED, h_layout=lay)
    got = B.grouped_gemm_swiglu_gather(c.x_k8, c.k, c.ss, c.d_codes, c.d_scales, c.gs,
                                       workspace=ws2, h_layout=lay)
    assert B.read_status(ws1) == B.MOE_OK and B.read_status(ws2) == B.MOE_OK
    np.testing.assert_array_equal(B.bits_from_bf16(got), B.bits_from_bf16(want))


def test_gather_matches_oracle(B):
    gs, k, K, I = GATHER_CASES["wide"]
    c = Case(B, gs, k, K, 2 * I, seed=6)
    h = B.grouped_gemm_swiglu_gather(c.x_k8, c.k, c.ss, c.d_codes, c.d_scales, c.gs)
    gsn, _, ss, _ = oracle.route_sort(c.ids, c.E)
    xs = oracle.gather(c.x, ss, c.k)
    y13, mag = oracle.grouped_gemm(xs, c.codes, c.scales, gsn)
    from parity_bounds import check_swiglu_from_gemm
    check_swiglu_from_gemm(B.bits_from_bf16(h), y13, mag, oracle.swiglu(y13), what="gather")


@pytest.mark.parametrize("name", ["split", "single", "wide", "layer_like"])
def test_scatter_writes_rows_in_slot_order(B, name):
    gs, k, K, I = GATHER_CASES[name]
    c = Case(B, gs, k, K, I, seed=8)
    want = B.grouped_gemm(c.x_sorted, c.d_codes, c.d_scales, c.gs,
                          act_layout=B.MOE_ACT_K8_INTERLEAVED)
    ws = c.ws()
    got = B.grouped_gemm_scatter(c.x_sorted, c.d_codes, c.d_scales, c.gs, c.ss, workspace=ws,
                                 act_layout=B.MOE_ACT_K8_INTERLEAVED)
    assert B.read_status(ws) == B.MOE_OK
    ss = c.ss.long()
    assert torch.equal(got[ss], want)


def test_scatter_skips_and_flags_rows_out_of_range(B):
    c = Case(B, [20, 0, 12, 4], 4, 256, 128, seed=9)
    out_row = c.ss.clone()
    out_row[3] = -1
    out_row[7] = out_row.numel() + 5
    sentinel = torch.full((out_row.numel(), 128), 7.0, device=DEV)
    ws = c.ws()
    B.grouped_gemm_scatter(c.x_sorted, c.d_codes, c.d_scales, c.gs, out_row, out=sentinel,
                           workspace=ws, act_layout=B.MOE_ACT_K8_INTERLEAVED)
    assert B.read_status(ws) == B.MOE_ERR_DATA
    want = B.grouped_gemm(c.x_sorted, c.d_codes, c.d_scales, c.gs,
                          act_layout=B.MOE_ACT_K8_INTERLEAVED)
    ok = torch.ones(out_row.numel(), dtype=torch.bool, device=DEV)
    ok[3] = ok[7] = False
    dst = out_row[ok].long()
    assert torch.equal(sentinel[dst], want[ok])
    # the rows that rows 3 and 7 should have written keep the sentinel
    assert torch.all(sentinel[c.ss[3].long()] == 7.0) and torch.all(sentinel[c.ss[7].long()] == 7.0)


def test_combine_slots_equals_combine(B):
    T, k, N, E = 50, 4, 384, 9
    rng = np.random.default_rng(5)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    ids[7, 2] = E + 3                       # one slot out of range
    gs, off, ss, s2r = B.route_sort(B.to_device(ids, DEV), E)[:4]
    y_sorted = torch.randn(T * k, N, device=DEV)
    w = torch.rand(T, k, device=DEV)
    want = B.combine(y_sorted, s2r, w)
    # slot order: slot s holds sorted row s2r[s]; the bad slot's row is garbage
    y_slots = torch.full((T * k, N), float("nan"), device=DEV)
    good = s2r >= 0
    y_slots[good] = y_sorted[s2r[good].long()]
    got = B.combine_slots(y_slots, s2r, w)
    assert torch.equal(got, want)
    got_bf16 = B.combine_slots(y_slots, s2r, w, out_dtype=torch.bfloat16)
    assert torch.equal(got_bf16, B.combine(y_sorted, s2r, w, out_dtype=torch.bfloat16))


@pytest.mark.parametrize("rows,hidden", [(1, 8), (37, 4096), (1000, 2048)])
def test_act_interleave_k8(B, rows, hidden):
    x = inputs.normal_bf16(1, 3, (rows, hidden))
    got = B.bits_from_bf16(B.act_interleave_k8(B.bf16_from_bits(x, DEV)))
    np.testing.assert_array_equal(got, k8_interleave(x))


def test_route_sort_token_order_k8_output(B):
    # x_layout MOE_ACT_K8_TOKEN_ORDER: x itself, interleaved, in token order;
    # the sort outputs are those of the plain route sort.
    T, k, E, H = 77, 3, 10, 512
    rng = np.random.default_rng(12)
    ids = B.to_device(rng.integers(0, E, (T, k)).astype(np.int32), DEV)
    x = inputs.normal_bf16(2, 5, (T, H))
    got = B.route_sort(ids, E, B.bf16_from_bits(x, DEV), x_layout=B.MOE_ACT_K8_TOKEN_ORDER)
    want = B.route_sort(ids, E)
    for a, b in zip(got[:4], want[:4]):
        assert torch.equal(a, b)
    assert got[4].shape == (T, H)
    np.testing.assert_array_equal(B.bits_from_bf16(got[4]), k8_interleave(x))
