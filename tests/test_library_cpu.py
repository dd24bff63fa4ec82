"""Host-side checks of the C ABI that need no GPU: the shared library builds,
loads, exports every entry point the header declares, and rejects bad
arguments before touching the device."""
import ctypes as C
import os
import re

import pytest

from fp4_weight_grouped_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = build_lib.build()
    return C.CDLL(path)


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_mxfp4.h")).read()
    return re.findall(r"MOE_API[^;(]*?\b(moe_\w+)\s*\(", src)


def test_header_declares_the_hot_path_calls():
    names = set(_declared())
    for n in ("moe_route_sort", "moe_mxfp4_grouped_gemm", "moe_swiglu", "moe_combine"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_symbol_list_matches_header():
    from fp4_weight_grouped_gb300 import binding
    assert set(binding.SYMBOLS) == set(_declared())


def test_status_strings(lib):
    lib.moe_status_string.restype = C.c_char_p
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(5) == b"MOE_ERR_TIMEOUT"


def test_workspace_bytes(lib):
    lib.moe_workspace_bytes.restype = C.c_size_t
    lib.moe_workspace_bytes.argtypes = [C.c_int32] * 3
    assert lib.moe_workspace_bytes(0, 6, 256) == 256
    # 49152 rows -> 48 chunks of 1024: 48*256*4 counts + 49152*4 ranks (256-byte rounded)
    assert lib.moe_workspace_bytes(8192, 6, 256) == 256 + 48 * 256 * 4 + 49152 * 4


def test_nvfp4_cast_workspace_and_host_checks(lib):
    lib.moe_nvfp4_cast_workspace_bytes.restype = C.c_size_t
    lib.moe_nvfp4_cast_workspace_bytes.argtypes = [C.c_int32]
    assert lib.moe_nvfp4_cast_workspace_bytes(1) == 512
    assert lib.moe_nvfp4_cast_workspace_bytes(256) == 256 + 1024
    f = lib.moe_mxfp4_to_nvfp4
    P = C.c_void_p
    f.argtypes = [P, C.c_int32, C.c_int32, C.c_int32, P, P, P, P, C.c_size_t, P]
    f.restype = C.c_int
    fake = P(4096)

    def call(s=fake, E=4, N=8, K=64, o=fake, w2=fake, oob=fake, ws=fake, wsb=1 << 12):
        return f(s, E, N, K, o, w2, oob, ws, wsb, None)

    INVALID = 1
    assert call(K=48) == INVALID            # K % 32
    assert call(K=0) == INVALID
    assert call(E=0) == INVALID
    assert call(E=65536) == INVALID         # one grid row per expert
    assert call(N=0) == INVALID
    assert call(s=None) == INVALID
    assert call(o=None) == INVALID
    assert call(w2=None) == INVALID
    assert call(oob=None) == INVALID
    assert call(oob=P(4100)) == INVALID     # uint64 counts need 8-byte alignment
    assert call(ws=P(4104)) == INVALID
    assert call(wsb=256 + 15) == INVALID    # E = 4 needs 256 + 256 bytes


def test_nvfp4_gemm_rejects_bad_arguments_on_host(lib):
    f = lib.moe_nvfp4_grouped_gemm
    P = C.c_void_p
    f.argtypes = [P, C.c_int, C.c_int64, C.c_int32, P, P, P, P, C.c_int32, C.c_int32, P, C.c_int, P,
                  C.c_size_t, P]
    f.restype = C.c_int
    fake = P(4096)

    def call(K=256, ws2=fake, s16=fake):
        return f(fake, 0, 8, K, fake, s16, ws2, fake, 4, 128, fake, 0, fake, 1 << 12, None)

    INVALID = 1
    assert call(ws2=None) == INVALID
    assert call(ws2=P(4098)) == INVALID     # f32 scales need 4-byte alignment
    assert call(s16=None) == INVALID
    assert call(K=48) == INVALID            # K % 32
    assert call(K=0) == INVALID


def test_gemm_rejects_bad_arguments_on_host(lib):
    f = lib.moe_mxfp4_grouped_gemm
    P = C.c_void_p
    f.argtypes = [P, C.c_int, C.c_int64, C.c_int32, P, P, P, C.c_int32, C.c_int32, P, C.c_int, P,
                  C.c_size_t, P]
    f.restype = C.c_int
    fake = P(4096)
    ok = dict(act=fake, lay=0, rows=32, K=256, codes=fake, scales=fake, gs=fake, E=8, N=512, out=fake,
              dt=0, ws=fake, wsb=256, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["act"], a["lay"], a["rows"], a["K"], a["codes"], a["scales"], a["gs"], a["E"],
                 a["N"], a["out"], a["dt"], a["ws"], a["wsb"], a["s"])

    INVALID = 1
    assert call(K=48) == INVALID            # K % 32
    assert call(K=0) == INVALID
    assert call(E=0) == INVALID
    assert call(E=1025) == INVALID
    assert call(N=0) == INVALID
    assert call(rows=-1) == INVALID
    assert call(codes=None) == INVALID
    assert call(scales=None) == INVALID
    assert call(gs=None) == INVALID
    assert call(ws=None) == INVALID
    assert call(wsb=255) == INVALID
    assert call(act=P(4098)) == INVALID     # TMA needs 16-byte aligned bases
    assert call(codes=P(4104)) == INVALID
    assert call(dt=7) == INVALID
    assert call(lay=2) == INVALID
    # No call here gets past the host checks: the pointers are not device memory,
    # so a call with valid arguments would reach a kernel launch on a GPU machine.


def test_route_sort_rejects_bad_arguments_on_host(lib):
    f = lib.moe_route_sort
    P = C.c_void_p
    f.argtypes = [P, C.c_int32, C.c_int32, C.c_int32, P, P, P, P, P, C.c_int32, P, C.c_int, P,
                  C.c_size_t, P]
    f.restype = C.c_int
    fake = P(4096)
    assert f(fake, 16, 7, 6, fake, fake, fake, fake, None, 0, None, 0, fake, 1 << 20, None) == 1   # k > E
    assert f(fake, 16, 2, 8, fake, fake, fake, fake, fake, 256, None, 0, fake, 1 << 20, None) == 1  # x, no x_sorted
    assert f(fake, 16, 2, 8, fake, fake, fake, fake, fake, 12, fake, 0, fake, 1 << 20, None) == 1   # hidden % 8
    assert f(fake, 16, 2, 8, fake, fake, fake, fake, None, 0, None, 0, fake, 100, None) == 1        # small ws
    assert f(fake, 16, 2, 8, fake, fake, fake, fake, None, 0, None, 5, fake, 1 << 20, None) == 1    # bad layout


def test_block_gemm_rejects_bad_block_on_host(lib):
    f = lib.moe_mxfp4_grouped_gemm_block
    P = C.c_void_p
    f.argtypes = [P, C.c_int, C.c_int64, C.c_int32, C.c_int32, P, P, P, C.c_int32, C.c_int32, P,
                  C.c_int, P, C.c_size_t, P]
    f.restype = C.c_int
    fake = P(4096)

    def call(K=1024, block=512):
        return f(fake, 0, 8, K, block, fake, fake, fake, 4, 128, fake, 0, fake, 1 << 12, None)

    assert call(block=64) == 1
    assert call(block=0) == 1
    assert call(K=768) == 1          # K % 512
    assert call(K=0) == 1
