"""Python binding of the C ABI in ``include/moe_mxfp4.h`` (argument marshalling
only).  Every compute step runs in the library's CUDA kernels; torch supplies
device memory (tensors) and the current CUDA stream.  If the shared library is
missing the calls raise: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

from . import build_lib

(MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DATA, MOE_ERR_TIMEOUT,
 MOE_ERR_CAPACITY) = range(7)
MOE_ROUTE_SORT_NOALLOC_SCRATCH_BYTES = 512 * 1024
MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_ROW_MAJOR, MOE_ACT_K8_INTERLEAVED, MOE_ACT_K8_TOKEN_ORDER = 0, 1, 2

SYMBOLS = (
    "moe_status_string", "moe_workspace_bytes", "moe_clear_status", "moe_read_status",
    "moe_route_sort", "moe_mxfp4_grouped_gemm", "moe_swiglu", "moe_combine", "moe_layer_forward",
    "moe_mxfp4_decode_expert", "moe_debug_bounded_wait", "moe_last_launch_count",
    "moe_route_sort_noalloc", "moe_nvfp4_cast_workspace_bytes", "moe_mxfp4_to_nvfp4",
    "moe_nvfp4_grouped_gemm", "moe_mxfp4_grouped_gemm_swiglu", "moe_mxfp4_grouped_gemm_block",
    "moe_mxfp4_grouped_gemm_swiglu_gather", "moe_mxfp4_grouped_gemm_scatter", "moe_combine_slots",
    "moe_act_interleave_k8", "moe_set_gemm_pairing",
)

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def library_path() -> str:
    return build_lib.LIB


def load(path: str | None = None):
    """Load the shared library (it must have been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or build_lib.LIB
            if not os.path.exists(p):
                raise RuntimeError(f"CUDA library not built: {p} (run __graft_entry__.build())")
            lib = C.CDLL(p)
            P, I32, I64, SZ, U64 = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t, C.c_uint64
            sig = {
                "moe_status_string": ([C.c_int], C.c_char_p),
                "moe_workspace_bytes": ([I32, I32, I32], SZ),
                "moe_clear_status": ([P, P], C.c_int),
                "moe_read_status": ([P, P], C.c_int),
                "moe_route_sort": ([P, I32, I32, I32, P, P, P, P, P, I32, P, C.c_int, P, SZ, P], C.c_int),
                "moe_route_sort_noalloc": ([P, I32, I32, I32, P, P, P, P, P, I32, P, C.c_int, P],
                                           C.c_int),
                "moe_mxfp4_grouped_gemm": ([P, C.c_int, I64, I32, P, P, P, I32, I32, P, C.c_int, P, SZ,
                                            P], C.c_int),
                "moe_mxfp4_grouped_gemm_block": ([P, C.c_int, I64, I32, I32, P, P, P, I32, I32, P,
                                                  C.c_int, P, SZ, P], C.c_int),
                "moe_mxfp4_grouped_gemm_swiglu": ([P, C.c_int, I64, I32, P, P, P, I32, I32, P,
                                                   C.c_int, P, SZ, P], C.c_int),
                "moe_mxfp4_grouped_gemm_swiglu_gather": ([P, I32, I32, P, I64, I32, P, P, P, I32,
                                                          I32, P, C.c_int, P, SZ, P], C.c_int),
                "moe_mxfp4_grouped_gemm_scatter": ([P, C.c_int, I64, I32, P, P, P, I32, I32, P, P,
                                                    C.c_int, P, SZ, P], C.c_int),
                "moe_combine_slots": ([P, P, P, I32, I32, I32, P, C.c_int, P], C.c_int),
                "moe_act_interleave_k8": ([P, I64, I32, P, P], C.c_int),
                "moe_set_gemm_pairing": ([I32], C.c_int),
                "moe_swiglu": ([P, C.c_int, I64, I32, P, C.c_int, P], C.c_int),
                "moe_combine": ([P, P, P, I32, I32, I32, P, C.c_int, P], C.c_int),
                "moe_layer_forward": ([P, P, P, I32, I32, I32, I32, I32, P, P, P, P, P,
                                       P, P, P, P, P, P, P, P, SZ, P], C.c_int),
                "moe_mxfp4_decode_expert": ([P, P, I32, I32, I32, I32, P, P, SZ, P], C.c_int),
                "moe_debug_bounded_wait": ([U64, P, SZ, P], C.c_int),
                "moe_last_launch_count": ([], I32),
                "moe_nvfp4_cast_workspace_bytes": ([I32], SZ),
                "moe_mxfp4_to_nvfp4": ([P, I32, I32, I32, P, P, P, P, SZ, P], C.c_int),
                "moe_nvfp4_grouped_gemm": ([P, C.c_int, I64, I32, P, P, P, P, I32, I32, P, C.c_int,
                                            P, SZ, P], C.c_int),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    try:
        return load().moe_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _dtype_code(dt) -> int:
    if dt == torch.float32:
        return MOE_F32
    if dt == torch.bfloat16:
        return MOE_BF16
    raise ValueError(f"unsupported dtype {dt}")


MOE_PAIRING_AUTO, MOE_PAIRING_OFF, MOE_PAIRING_ON = 0, 1, 2


def set_gemm_pairing(mode: int):
    """CTA pairs for bands over 32 rows: MOE_PAIRING_AUTO / _OFF / _ON (process-wide)."""
    _check(load().moe_set_gemm_pairing(int(mode)), "moe_set_gemm_pairing")


def last_launch_count() -> int:
    return int(load().moe_last_launch_count())


# ---------------------------------------------------------------- workspace

def workspace_bytes(T: int, k: int, E: int) -> int:
    return int(load().moe_workspace_bytes(T, k, E))


def make_workspace(T: int, k: int, E: int, device="cuda", stream=None) -> torch.Tensor:
    ws = torch.empty(workspace_bytes(T, k, E), dtype=torch.uint8, device=device)
    clear_status(ws, stream)
    return ws


def clear_status(workspace: torch.Tensor, stream=None):
    _check(load().moe_clear_status(_ptr(workspace), _stream(stream)), "moe_clear_status")


def read_status(workspace: torch.Tensor, stream=None) -> int:
    return int(load().moe_read_status(_ptr(workspace), _stream(stream)))


# ---------------------------------------------------------------- operations

def route_sort(topk_ids: torch.Tensor, E: int, x: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, out=None, stream=None,
               x_layout: int = MOE_ACT_ROW_MAJOR):
    """Returns (group_sizes[E], group_offsets[E+1], sorted_slot[T*k],
    slot_to_row[T*k], x_sorted or None); x_sorted in `x_layout` order
    (MOE_ACT_K8_TOKEN_ORDER: x itself [T, hidden] in the K8 order)."""
    T, k = topk_ids.shape
    dev = topk_ids.device
    rows = T * k
    if out is None:
        gs = torch.empty(E, dtype=torch.int32, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        ss = torch.empty(rows, dtype=torch.int32, device=dev)
        s2r = torch.empty(rows, dtype=torch.int32, device=dev)
        xs_rows = T if x_layout == MOE_ACT_K8_TOKEN_ORDER else rows
        xs = None if x is None else torch.empty((xs_rows, x.shape[1]), dtype=x.dtype, device=dev)
    else:
        gs, off, ss, s2r, xs = out
    if workspace is None:
        workspace = make_workspace(T, k, E, dev, stream)
    hidden = 0 if x is None else x.shape[1]
    rc = load().moe_route_sort(_ptr(topk_ids), T, k, E, _ptr(gs), _ptr(off), _ptr(ss), _ptr(s2r),
                               _ptr(x), hidden, _ptr(xs), x_layout, _ptr(workspace),
                               workspace.numel(), _stream(stream))
    _check(rc, "moe_route_sort")
    return gs, off, ss, s2r, xs


def route_sort_noalloc(topk_ids: torch.Tensor, E: int, out, x: torch.Tensor | None = None,
                       stream=None, x_layout: int = MOE_ACT_ROW_MAJOR):
    """Route sort through the fixed-capacity entry point, for callers that must
    not allocate at the point of the call.  `out` = (group_sizes, group_offsets,
    sorted_slot, slot_to_row, x_sorted or None) must already exist: this wrapper
    creates no tensor, and the library call uses its own static scratch instead
    of a workspace.  Raises MoeError(MOE_ERR_CAPACITY) when the problem needs
    more than MOE_ROUTE_SORT_NOALLOC_SCRATCH_BYTES of scratch."""
    T, k = topk_ids.shape
    gs, off, ss, s2r, xs = out
    hidden = 0 if x is None else x.shape[1]
    rc = load().moe_route_sort_noalloc(_ptr(topk_ids), T, k, E, _ptr(gs), _ptr(off), _ptr(ss),
                                       _ptr(s2r), _ptr(x), hidden, _ptr(xs), x_layout,
                                       _stream(stream))
    _check(rc, "moe_route_sort_noalloc")
    return out


def grouped_gemm(act: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                 group_sizes: torch.Tensor, out: torch.Tensor | None = None,
                 out_dtype=torch.float32, workspace: torch.Tensor | None = None, stream=None,
                 act_layout: int = MOE_ACT_ROW_MAJOR):
    """act bf16 [rows, K] (row-major or K8-interleaved); codes uint8 [E, N, K/2];
    scales uint8 [E, N, K/32]; group_sizes int32 [E] -> out [rows, N] (f32 or bf16)."""
    rows, K = act.shape
    E, N, _ = codes.shape
    if out is None:
        out = torch.empty((rows, N), dtype=out_dtype, device=act.device)
    if workspace is None:
        workspace = make_workspace(0, 1, 1, act.device, stream)
    rc = load().moe_mxfp4_grouped_gemm(_ptr(act), act_layout, rows, K, _ptr(codes), _ptr(scales),
                                       _ptr(group_sizes), E, N, _ptr(out), _dtype_code(out.dtype),
                                       _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "moe_mxfp4_grouped_gemm")
    return out


def grouped_gemm_block(act: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                       group_sizes: torch.Tensor, scale_block: int, out: torch.Tensor | None = None,
                       out_dtype=torch.float32, workspace: torch.Tensor | None = None, stream=None,
                       act_layout: int = MOE_ACT_ROW_MAJOR):
    """grouped_gemm with one E8M0 scale per `scale_block` (32 or 512)
    consecutive k: scales uint8 [E, N, K / scale_block]."""
    rows, K = act.shape
    E, N, _ = codes.shape
    if out is None:
        out = torch.empty((rows, N), dtype=out_dtype, device=act.device)
    if workspace is None:
        workspace = make_workspace(0, 1, 1, act.device, stream)
    rc = load().moe_mxfp4_grouped_gemm_block(_ptr(act), act_layout, rows, K, int(scale_block),
                                             _ptr(codes), _ptr(scales), _ptr(group_sizes), E, N,
                                             _ptr(out), _dtype_code(out.dtype), _ptr(workspace),
                                             workspace.numel(), _stream(stream))
    _check(rc, "moe_mxfp4_grouped_gemm_block")
    return out


def grouped_gemm_swiglu(act: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                        group_sizes: torch.Tensor, out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None,
                        act_layout: int = MOE_ACT_ROW_MAJOR, h_layout: int = MOE_ACT_ROW_MAJOR):
    """w13 grouped GEMM with SwiGLU in its epilogue.  act bf16 [rows, K]; codes
    uint8 [E, 2I, K/2] and scales uint8 [E, 2I, K/32] with gate rows [0, I) and
    up rows [I, 2I); group_sizes int32 [E] -> h bf16 [rows, I] in `h_layout`."""
    rows, K = act.shape
    E, two_i, _ = codes.shape
    I = two_i // 2
    if out is None:
        out = torch.empty((rows, I), dtype=torch.bfloat16, device=act.device)
    if workspace is None:
        workspace = make_workspace(0, 1, 1, act.device, stream)
    rc = load().moe_mxfp4_grouped_gemm_swiglu(_ptr(act), act_layout, rows, K, _ptr(codes),
                                              _ptr(scales), _ptr(group_sizes), E, I, _ptr(out),
                                              h_layout, _ptr(workspace), workspace.numel(),
                                              _stream(stream))
    _check(rc, "moe_mxfp4_grouped_gemm_swiglu")
    return out


def grouped_gemm_swiglu_gather(x_k8: torch.Tensor, top_k: int, sorted_slot: torch.Tensor,
                               codes: torch.Tensor, scales: torch.Tensor,
                               group_sizes: torch.Tensor, out: torch.Tensor | None = None,
                               workspace: torch.Tensor | None = None, stream=None,
                               h_layout: int = MOE_ACT_ROW_MAJOR):
    """grouped_gemm_swiglu with the activation rows gathered in the load: sorted
    row r reads row sorted_slot[r] // top_k of x_k8 bf16 [T, K] (K8-interleaved);
    -> h bf16 [rows, I], rows = sorted_slot.numel()."""
    T, K = x_k8.shape
    rows = sorted_slot.numel()
    E, two_i, _ = codes.shape
    I = two_i // 2
    if out is None:
        out = torch.empty((rows, I), dtype=torch.bfloat16, device=x_k8.device)
    if workspace is None:
        workspace = make_workspace(0, 1, 1, x_k8.device, stream)
    rc = load().moe_mxfp4_grouped_gemm_swiglu_gather(
        _ptr(x_k8), T, int(top_k), _ptr(sorted_slot), rows, K, _ptr(codes), _ptr(scales),
        _ptr(group_sizes), E, I, _ptr(out), h_layout, _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check(rc, "moe_mxfp4_grouped_gemm_swiglu_gather")
    return out


def grouped_gemm_scatter(act: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                         group_sizes: torch.Tensor, out_row: torch.Tensor,
                         out: torch.Tensor | None = None, out_dtype=torch.float32,
                         workspace: torch.Tensor | None = None, stream=None,
                         act_layout: int = MOE_ACT_ROW_MAJOR):
    """grouped_gemm writing sorted row r to row out_row[r] of out [rows, N]."""
    rows, K = act.shape
    E, N, _ = codes.shape
    if out is None:
        out = torch.empty((rows, N), dtype=out_dtype, device=act.device)
    if workspace is None:
        workspace = make_workspace(0, 1, 1, act.device, stream)
    rc = load().moe_mxfp4_grouped_gemm_scatter(_ptr(act), act_layout, rows, K, _ptr(codes),
                                               _ptr(scales), _ptr(group_sizes), E, N,
                                               _ptr(out_row), _ptr(out), _dtype_code(out.dtype),
                                               _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "moe_mxfp4_grouped_gemm_scatter")
    return out


def act_interleave_k8(x: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    """bf16 [rows, hidden] -> the same rows in the K8-interleaved order."""
    rows, hidden = x.shape
    if out is None:
        out = torch.empty_like(x)
    rc = load().moe_act_interleave_k8(_ptr(x), rows, hidden, _ptr(out), _stream(stream))
    _check(rc, "moe_act_interleave_k8")
    return out


def nvfp4_grouped_gemm(act: torch.Tensor, codes: torch.Tensor, scales16: torch.Tensor,
                       weight_scale_2: torch.Tensor, group_sizes: torch.Tensor,
                       out: torch.Tensor | None = None, out_dtype=torch.float32,
                       workspace: torch.Tensor | None = None, stream=None,
                       act_layout: int = MOE_ACT_ROW_MAJOR):
    """act bf16 [rows, K]; codes uint8 [E, N, K/2]; scales16 uint8 [E, N, K/16]
    (E4M3); weight_scale_2 f32 [E]; group_sizes int32 [E] -> out [rows, N]."""
    rows, K = act.shape
    E, N, _ = codes.shape
    if out is None:
        out = torch.empty((rows, N), dtype=out_dtype, device=act.device)
    if workspace is None:
        workspace = make_workspace(0, 1, 1, act.device, stream)
    rc = load().moe_nvfp4_grouped_gemm(_ptr(act), act_layout, rows, K, _ptr(codes), _ptr(scales16),
                                       _ptr(weight_scale_2), _ptr(group_sizes), E, N, _ptr(out),
                                       _dtype_code(out.dtype), _ptr(workspace), workspace.numel(),
                                       _stream(stream))
    _check(rc, "moe_nvfp4_grouped_gemm")
    return out


def swiglu(gu: torch.Tensor, out: torch.Tensor | None = None, stream=None,
           layout: int = MOE_ACT_ROW_MAJOR):
    rows, two_i = gu.shape
    I = two_i // 2
    if out is None:
        out = torch.empty((rows, I), dtype=torch.bfloat16, device=gu.device)
    rc = load().moe_swiglu(_ptr(gu), _dtype_code(gu.dtype), rows, I, _ptr(out), layout,
                           _stream(stream))
    _check(rc, "moe_swiglu")
    return out


def combine(y: torch.Tensor, slot_to_row: torch.Tensor, topk_w: torch.Tensor,
            out: torch.Tensor | None = None, out_dtype=torch.float32, stream=None):
    T, k = topk_w.shape
    N = y.shape[1]
    if out is None:
        out = torch.empty((T, N), dtype=out_dtype, device=y.device)
    rc = load().moe_combine(_ptr(y), _ptr(slot_to_row), _ptr(topk_w), T, k, N, _ptr(out),
                            _dtype_code(out.dtype), _stream(stream))
    _check(rc, "moe_combine")
    return out


def combine_slots(y: torch.Tensor, slot_to_row: torch.Tensor, topk_w: torch.Tensor,
                  out: torch.Tensor | None = None, out_dtype=torch.float32, stream=None):
    """combine with y f32 [T*k, N] in slot order (slot_to_row marks valid slots)."""
    T, k = topk_w.shape
    N = y.shape[1]
    if out is None:
        out = torch.empty((T, N), dtype=out_dtype, device=y.device)
    rc = load().moe_combine_slots(_ptr(y), _ptr(slot_to_row), _ptr(topk_w), T, k, N, _ptr(out),
                                  _dtype_code(out.dtype), _stream(stream))
    _check(rc, "moe_combine_slots")
    return out


class LayerBuffers:
    """Caller-owned intermediates of one layer pass (allocated once, reused)."""

    def __init__(self, T: int, k: int, E: int, hidden: int, inter: int, device="cuda"):
        rows = T * k
        i32 = dict(dtype=torch.int32, device=device)
        self.group_sizes = torch.empty(E, **i32)
        self.group_offsets = torch.empty(E + 1, **i32)
        self.sorted_slot = torch.empty(rows, **i32)
        self.slot_to_row = torch.empty(rows, **i32)
        self.x_sorted = torch.empty((rows, hidden), dtype=torch.bfloat16, device=device)
        self.h = torch.empty((rows, inter), dtype=torch.bfloat16, device=device)
        self.y2 = torch.empty((rows, hidden), dtype=torch.float32, device=device)
        self.out = torch.empty((T, hidden), dtype=torch.float32, device=device)
        self.workspace = make_workspace(T, k, E, device)


def layer_forward(x, topk_ids, topk_w, w13_codes, w13_scales, w2_codes, w2_scales,
                  buffers: LayerBuffers, stream=None):
    T, k = topk_ids.shape
    E, two_i, hidden_half = w13_codes.shape
    hidden, inter = 2 * hidden_half, two_i // 2
    b = buffers
    rc = load().moe_layer_forward(
        _ptr(x), _ptr(topk_ids), _ptr(topk_w), T, k, E, hidden, inter,
        _ptr(w13_codes), _ptr(w13_scales), _ptr(w2_codes), _ptr(w2_scales), _ptr(b.out),
        _ptr(b.group_sizes), _ptr(b.group_offsets), _ptr(b.sorted_slot), _ptr(b.slot_to_row),
        _ptr(b.x_sorted), _ptr(b.h), _ptr(b.y2), _ptr(b.workspace),
        b.workspace.numel(), _stream(stream))
    _check(rc, "moe_layer_forward")
    return b.out


def decode_expert(codes: torch.Tensor, scales: torch.Tensor, e: int,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    E, N, Kh = codes.shape
    K = 2 * Kh
    out = torch.empty((N, K), dtype=torch.bfloat16, device=codes.device)
    if workspace is None:
        workspace = make_workspace(0, 1, 1, codes.device, stream)
    rc = load().moe_mxfp4_decode_expert(_ptr(codes), _ptr(scales), E, N, K, e, _ptr(out),
                                        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "moe_mxfp4_decode_expert")
    return out


def mxfp4_to_nvfp4(scales: torch.Tensor, out=None, workspace: torch.Tensor | None = None,
                   stream=None):
    """Lossless MXFP4 -> NVFP4 scale cast.  scales uint8 [E, N, K/32] ->
    (e4m3 uint8 [E, N, K/16], weight_scale_2 f32 [E], out_of_range int64 [E]);
    `out` may hold those three tensors already (out_of_range holds the uint64
    counts of the C call, which never exceed 2^63)."""
    E, N, Kb = scales.shape
    dev = scales.device
    if out is None:
        out = (torch.empty((E, N, 2 * Kb), dtype=torch.uint8, device=dev),
               torch.empty(E, dtype=torch.float32, device=dev),
               torch.empty(E, dtype=torch.int64, device=dev))
    e4m3, ws2, oob = out
    if workspace is None:
        workspace = torch.empty(int(load().moe_nvfp4_cast_workspace_bytes(E)), dtype=torch.uint8,
                                device=dev)
        clear_status(workspace, stream)
    rc = load().moe_mxfp4_to_nvfp4(_ptr(scales), E, N, 32 * Kb, _ptr(e4m3), _ptr(ws2), _ptr(oob),
                                   _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "moe_mxfp4_to_nvfp4")
    return out


def debug_bounded_wait(limit_ns: int, workspace: torch.Tensor, stream=None):
    rc = load().moe_debug_bounded_wait(int(limit_ns), _ptr(workspace), workspace.numel(),
                                       _stream(stream))
    _check(rc, "moe_debug_bounded_wait")


# ---------------------------------------------------------------- marshalling

def bf16_from_bits(bits, device="cuda") -> torch.Tensor:
    """numpy uint16 bf16 patterns -> device bf16 tensor (bit-exact)."""
    import numpy as np
    a = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a).to(device).view(torch.bfloat16)


def bits_from_bf16(t: torch.Tensor):
    """device bf16 tensor -> numpy uint16 bit patterns."""
    import numpy as np
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_device(a, device="cuda") -> torch.Tensor:
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)
