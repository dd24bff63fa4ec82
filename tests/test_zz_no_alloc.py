"""The fixed-capacity route sort (moe_route_sort_noalloc) against the
workspace route sort (moe_route_sort).

The file name sorts last so that these tests also run after every other test
of the suite; each test passes on its own as well.  Route sort is integer
work, so the bar is bit-exact equality with the workspace entry point (which
the parity suite holds bit-exact to the oracle).
"""
import ctypes as C

import numpy as np
import pytest

from fp4_weight_grouped_gb300 import build_lib, inputs

SCRATCH_MAX = 512 * 1024


def _scratch_bytes(T, k, E):
    rows = T * k
    chunks = (rows + 1023) // 1024
    up = lambda b: (b + 255) // 256 * 256
    return up(chunks * E * 4) + up(rows * 4)


# ------------------------------------------------------------ host side (CPU)

def test_capacity_is_checked_on_the_host():
    lib = C.CDLL(build_lib.build())
    f = lib.moe_route_sort_noalloc
    P, I32 = C.c_void_p, C.c_int32
    f.argtypes = [P, I32, I32, I32, P, P, P, P, P, I32, P, C.c_int, P]
    f.restype = C.c_int
    fake = P(4096)
    # 17408 * 6 = 104448 slots at E = 256: 522240 bytes of scratch, fits (the
    # GPU test below runs it; here only calls rejected on the host are made,
    # because the pointers are not device memory).
    assert _scratch_bytes(17408, 6, 256) <= SCRATCH_MAX
    # One more 1024-slot chunk does not.
    assert _scratch_bytes(17408 + 171, 6, 256) > SCRATCH_MAX
    assert f(fake, 17408 + 171, 6, 256, fake, fake, fake, fake, None, 0, None, 0, None) == 6
    # Argument errors come before the capacity check.
    assert f(fake, 17408 + 171, 7, 6, fake, fake, fake, fake, None, 0, None, 0, None) == 1
    lib.moe_status_string.restype = C.c_char_p
    assert lib.moe_status_string(6) == b"MOE_ERR_CAPACITY"


# ------------------------------------------------------------------ GPU side

@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as g
    g.build()
    from fp4_weight_grouped_gb300 import binding
    binding.load()
    return binding


def _outputs(torch, T, k, E, hidden):
    rows = T * k
    dev = "cuda"
    return (torch.full((E,), -7, dtype=torch.int32, device=dev),
            torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            torch.full((rows,), -7, dtype=torch.int32, device=dev),
            torch.full((rows,), -7, dtype=torch.int32, device=dev),
            None if hidden == 0 else torch.zeros((rows, hidden), dtype=torch.bfloat16, device=dev))


def _assert_same(torch, got, want):
    for g, w in zip(got, want):
        if w is None:
            assert g is None
        else:
            assert torch.equal(g, w)


@pytest.mark.gpu
def test_two_consecutive_calls_match_the_workspace_route_sort(B):
    torch = pytest.importorskip("torch")
    E, k, hidden = 256, 6, 512
    ids_a = inputs.route_zipf(11, 4096, E, k)        # 24 chunks, skewed, 20 experts unused
    ids_b = inputs.route_uniform(12, 1500, E, k)     # ragged last chunk
    x_a = B.bf16_from_bits(inputs.normal_bf16(11, 7, (4096, hidden)), "cuda")
    x_b = B.bf16_from_bits(inputs.normal_bf16(12, 7, (1500, hidden)), "cuda")
    d_a, d_b = B.to_device(ids_a, "cuda"), B.to_device(ids_b, "cuda")
    out_a = _outputs(torch, 4096, k, E, hidden)
    out_b = _outputs(torch, 1500, k, E, hidden)
    torch.cuda.synchronize()
    before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    B.route_sort_noalloc(d_a, E, out_a, x=x_a, x_layout=B.MOE_ACT_K8_INTERLEAVED)
    B.route_sort_noalloc(d_b, E, out_b, x=x_b)
    torch.cuda.synchronize()
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == before
    want_a = B.route_sort(d_a, E, x_a, x_layout=B.MOE_ACT_K8_INTERLEAVED)
    want_b = B.route_sort(d_b, E, x_b)
    torch.cuda.synchronize()
    _assert_same(torch, out_a, want_a)
    _assert_same(torch, out_b, want_b)


@pytest.mark.gpu
def test_largest_problem_that_fits(B):
    torch = pytest.importorskip("torch")
    T, k, E = 17408, 6, 256
    assert _scratch_bytes(T, k, E) <= SCRATCH_MAX
    ids = inputs.route_logits(13, T, E, k)[0]
    d = B.to_device(ids, "cuda")
    out = _outputs(torch, T, k, E, 0)
    B.route_sort_noalloc(d, E, out)
    want = B.route_sort(d, E)
    torch.cuda.synchronize()
    _assert_same(torch, out[:4], want[:4])


@pytest.mark.gpu
def test_over_capacity_raises_and_writes_nothing(B):
    torch = pytest.importorskip("torch")
    T, k, E = 17408 + 171, 6, 256
    ids = inputs.route_uniform(14, T, E, k)
    out = _outputs(torch, T, k, E, 0)
    with pytest.raises(B.MoeError) as err:
        B.route_sort_noalloc(B.to_device(ids, "cuda"), E, out)
    assert err.value.status == B.MOE_ERR_CAPACITY
    torch.cuda.synchronize()
    assert bool((out[1] == -7).all())


@pytest.mark.gpu
def test_bad_id_shows_as_missing_rows(B):
    torch = pytest.importorskip("torch")
    E, k = 64, 4
    ids = inputs.route_uniform(15, 300, E, k)
    ids[17, 2] = E
    out = _outputs(torch, 300, k, E, 0)
    B.route_sort_noalloc(B.to_device(ids, "cuda"), E, out)
    torch.cuda.synchronize()
    assert int(out[1][E]) == 300 * k - 1
