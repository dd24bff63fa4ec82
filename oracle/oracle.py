"""ctypes wrapper of the C oracle in ``oracle.c`` (test infrastructure only).

The shared object is built with the system C compiler into ``oracle/_build``;
``build()`` is idempotent and is also called by the repository's build step.
All floating-point results are float64.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O3", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared",
                        "-pthread", _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            P, L, I = C.c_void_p, C.c_long, C.c_int
            lib.oracle_e2m1_value.argtypes = [I]
            lib.oracle_e2m1_value.restype = C.c_double
            lib.oracle_double_to_bf16.argtypes = [C.c_double]
            lib.oracle_double_to_bf16.restype = C.c_uint16
            lib.oracle_bf16_to_double.argtypes = [C.c_uint16]
            lib.oracle_bf16_to_double.restype = C.c_double
            lib.oracle_decode_expert_bf16.argtypes = [P, P, L, L, L, L, P]
            lib.oracle_decode_expert_bf16.restype = I
            lib.oracle_route_sort.argtypes = [P, L, L, L, P, P, P, P]
            lib.oracle_route_sort.restype = I
            lib.oracle_gather.argtypes = [P, L, P, L, L, P]
            lib.oracle_gather.restype = None
            lib.oracle_grouped_gemm.argtypes = [P, L, L, P, P, P, L, L, P, P, I]
            lib.oracle_grouped_gemm.restype = I
            lib.oracle_grouped_gemm_block.argtypes = [P, L, L, L, P, P, P, L, L, P, P, I]
            lib.oracle_grouped_gemm_block.restype = I
            lib.oracle_grouped_gemm_sampled.argtypes = [P, L, L, P, P, P, L, L, P, P, L, P, P, I]
            lib.oracle_grouped_gemm_sampled.restype = I
            lib.oracle_swiglu.argtypes = [P, L, L, P]
            lib.oracle_swiglu.restype = None
            lib.oracle_combine.argtypes = [P, L, P, P, L, L, P, P]
            lib.oracle_combine.restype = None
            lib.oracle_e4m3_value.argtypes = [I]
            lib.oracle_e4m3_value.restype = C.c_double
            lib.oracle_mxfp4_to_nvfp4.argtypes = [P, L, L, L, P, P, P]
            lib.oracle_mxfp4_to_nvfp4.restype = I
            lib.oracle_nvfp4_grouped_gemm.argtypes = [P, L, L, P, P, P, P, L, L, P, P, I]
            lib.oracle_nvfp4_grouped_gemm.restype = I
            lib.oracle_threads_used.argtypes = []
            lib.oracle_threads_used.restype = I
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def threads_used() -> int:
    """Worker threads the last parallel oracle call ran on."""
    return _load().oracle_threads_used()


def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def double_to_bf16(x: float) -> int:
    return int(_load().oracle_double_to_bf16(float(x)))


def bf16_to_double(b: int) -> float:
    return float(_load().oracle_bf16_to_double(int(b)))


def decode_expert_bf16(codes: np.ndarray, scales: np.ndarray, e: int) -> np.ndarray:
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    E, N, Kh = codes.shape
    K = 2 * Kh
    out = np.empty((N, K), dtype=np.uint16)
    if _load().oracle_decode_expert_bf16(_p(codes), _p(scales), E, N, K, e, _p(out)):
        raise ValueError("bad expert index or scale byte > 252")
    return out


def route_sort(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    rows = T * k
    gs = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    ss = np.empty(rows, np.int32)
    s2r = np.empty(rows, np.int32)
    if _load().oracle_route_sort(_p(ids), T, k, E, _p(gs), _p(off), _p(ss), _p(s2r)):
        raise ValueError("expert id out of range")
    return gs, off, ss, s2r


def gather(x: np.ndarray, sorted_slot: np.ndarray, k: int) -> np.ndarray:
    x, ss = _c(x, np.uint16), _c(sorted_slot, np.int32)
    out = np.empty((ss.shape[0], x.shape[1]), np.uint16)
    _load().oracle_gather(_p(x), x.shape[1], _p(ss), ss.shape[0], k, _p(out))
    return out


def grouped_gemm(act, codes, scales, group_sizes, n_threads: int = 0, with_abs: bool = True):
    """Returns (out[rows, N], abs[rows, N]) in float64."""
    act = _c(act, np.uint16)
    codes, scales, gs = _c(codes, np.uint8), _c(scales, np.uint8), _c(group_sizes, np.int32)
    rows, K = act.shape
    E, N, _ = codes.shape
    out = np.zeros((rows, N), np.float64)
    mag = np.zeros((rows, N), np.float64) if with_abs else None
    rc = _load().oracle_grouped_gemm(_p(act), rows, K, _p(codes), _p(scales), _p(gs), E, N, _p(out),
                                     _p(mag) if with_abs else None, n_threads)
    if rc:
        raise ValueError("sum(group_sizes) != rows, a negative size, or a scale byte > 252")
    return out, mag


def grouped_gemm_block(act, codes, scales, group_sizes, block: int, n_threads: int = 0,
                       with_abs: bool = True):
    """The grouped GEMM with one E8M0 scale per `block` consecutive k (32 or
    512): scales uint8 [E, N, K/block].  Returns (out[rows, N], abs[rows, N])."""
    act = _c(act, np.uint16)
    codes, scales, gs = _c(codes, np.uint8), _c(scales, np.uint8), _c(group_sizes, np.int32)
    rows, K = act.shape
    E, N, _ = codes.shape
    out = np.zeros((rows, N), np.float64)
    mag = np.zeros((rows, N), np.float64) if with_abs else None
    rc = _load().oracle_grouped_gemm_block(_p(act), rows, K, int(block), _p(codes), _p(scales),
                                           _p(gs), E, N, _p(out), _p(mag) if with_abs else None,
                                           n_threads)
    if rc:
        raise ValueError("bad block, K % block, sizes, or a scale byte > 252")
    return out, mag


def grouped_gemm_sampled(act, codes, scales, group_sizes, srow, scol, n_threads: int = 0):
    act = _c(act, np.uint16)
    codes, scales, gs = _c(codes, np.uint8), _c(scales, np.uint8), _c(group_sizes, np.int32)
    srow, scol = _c(srow, np.int64), _c(scol, np.int64)
    rows, K = act.shape
    E, N, _ = codes.shape
    out = np.zeros(srow.shape[0], np.float64)
    mag = np.zeros(srow.shape[0], np.float64)
    rc = _load().oracle_grouped_gemm_sampled(_p(act), rows, K, _p(codes), _p(scales), _p(gs), E, N,
                                             _p(srow), _p(scol), srow.shape[0], _p(out), _p(mag),
                                             n_threads)
    if rc:
        raise ValueError("bad sizes, sample index or scale byte")
    return out, mag


def swiglu(gu: np.ndarray) -> np.ndarray:
    """gu float [rows, 2I] -> bf16 bits [rows, I]."""
    gu = _c(gu, np.float64)
    rows, two_i = gu.shape
    I = two_i // 2
    h = np.empty((rows, I), np.uint16)
    _load().oracle_swiglu(_p(gu), rows, I, _p(h))
    return h


def combine(y, slot_to_row, topk_w):
    """y float [rows, N], slot_to_row int [T*k], topk_w float32 [T, k] ->
    (out[T, N], abs[T, N]) in float64."""
    y = _c(y, np.float64)
    s2r = _c(slot_to_row, np.int32)
    w = _c(topk_w, np.float32)
    T, k = w.shape
    N = y.shape[1]
    out = np.empty((T, N), np.float64)
    mag = np.empty((T, N), np.float64)
    _load().oracle_combine(_p(y), N, _p(s2r), _p(w), T, k, _p(out), _p(mag))
    return out, mag


def e4m3_value(byte: int) -> float:
    return _load().oracle_e4m3_value(int(byte))


def mxfp4_to_nvfp4(scales: np.ndarray):
    """scales uint8 [E, N, K/32] (E8M0) -> (e4m3 uint8 [E, N, K/16],
    weight_scale_2 float64 [E], out_of_range int64 [E])."""
    scales = _c(scales, np.uint8)
    E, N, nb = scales.shape
    e4m3 = np.empty((E, N, 2 * nb), np.uint8)
    ws2 = np.empty(E, np.float64)
    oob = np.empty(E, np.int64)
    if _load().oracle_mxfp4_to_nvfp4(_p(scales), E, N, 32 * nb, _p(e4m3), _p(ws2), _p(oob)):
        raise ValueError("scale byte 255 (E8M0 NaN)")
    return e4m3, ws2, oob


def nvfp4_grouped_gemm(act, codes, scales16, weight_scale_2, group_sizes, n_threads: int = 0,
                       with_abs: bool = True):
    """NVFP4 W4A16 grouped GEMM in float64: codes uint8 [E, N, K/2], scales16
    uint8 [E, N, K/16] (E4M3), weight_scale_2 float32 [E].  Returns
    (out[rows, N], abs[rows, N] or None)."""
    act = _c(act, np.uint16)
    codes, s16 = _c(codes, np.uint8), _c(scales16, np.uint8)
    ws2, gs = _c(weight_scale_2, np.float32), _c(group_sizes, np.int32)
    rows, K = act.shape
    E, N, _ = codes.shape
    out = np.zeros((rows, N), np.float64)
    mag = np.zeros((rows, N), np.float64) if with_abs else None
    rc = _load().oracle_nvfp4_grouped_gemm(_p(act), rows, K, _p(codes), _p(s16), _p(ws2), _p(gs), E,
                                           N, _p(out), _p(mag) if with_abs else None, n_threads)
    if rc:
        raise ValueError("K % 16, sum(group_sizes) != rows, a negative size, or a NaN E4M3 scale")
    return out, mag
