"""Seeded synthetic inputs shaped like the MoE workloads of "Running DeepSeek V4
Flash on TPU v6" (section 1, "Four bits that v6e can't hold": 256 routed experts,
top-6 routing, w13 with K = N = 4096, w2 with K = 2048, N = 4096).

This module only draws random numbers and packs them into the byte layouts the
library consumes.  It holds no step of the method itself: no e2m1 decode, no
scaling, no sort, no matmul, no combine.  Both the CPU oracle (under ``oracle/``)
and the CUDA path take their inputs from here, and from nowhere else.

Layouts (all little-endian, C order):
  codes   uint8 [E, N, K/2]   two e2m1 nibbles per byte, element 2j in bits 0-3
  scales  uint8 [E, N, K/32]  E8M0 exponent bytes, 127 = 2^0
  act     uint16 [rows, K]    bfloat16 bit patterns
  ids     int32 [T, k]        routed expert per (token, choice)
  topk_w  float32 [T, k]      router weights
"""
from __future__ import annotations

import numpy as np

# Stream tags keep each tensor's random stream independent of the others, so a
# caller can regenerate one tensor without drawing the rest.
_TAG_ROUTE, _TAG_ACT, _TAG_W13, _TAG_W2, _TAG_X, _TAG_GATE, _TAG_SCALES, _TAG_NV = 1, 2, 3, 4, 5, 6, 7, 8

CONFIGS = {
    # Tiny MXFP4 grouped GEMM: E=8, top-2, T=16 (32 rows), K=256, N=512,
    # E8M0 exponents in [-8, -4], expert 5 forced empty.
    "tiny": dict(kind="gemm", E=8, k=2, T=16, K=256, N=512, exp=(-8, -4),
                 routing="uniform", empty=(5,), act="normal"),
    # Decode w13: E=256, top-6, T=64 (384 rows), K=N=4096.
    "decode_w13": dict(kind="gemm", E=256, k=6, T=64, K=4096, N=4096, exp=(-10, -2),
                       routing="uniform", empty=(), act="normal"),
    # Decode w2: E=256, top-6, T=256 (1536 rows), K=2048, N=4096, activations
    # shaped like the output of a SwiGLU of N(0,1) pairs.
    "decode_w2": dict(kind="gemm", E=256, k=6, T=256, K=2048, N=4096, exp=(-10, -2),
                      routing="uniform", empty=(), act="swiglu_pairs"),
    # Prefill w13: E=256, top-6, T=4096 (24576 rows), K=N=4096, Zipf(1.1)
    # expert popularity with 20 experts never chosen.
    "prefill_w13": dict(kind="gemm", E=256, k=6, T=4096, K=4096, N=4096, exp=(-10, -2),
                        routing="zipf", empty=(), act="normal"),
    # Full MoE layer: T=8192, hidden 4096, 256 experts top-6, intermediate 2048.
    "layer": dict(kind="layer", E=256, k=6, T=8192, hidden=4096, inter=2048, exp=(-10, -2),
                  routing="logits"),
}


def _rng(seed: int, tag: int, *extra: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, *extra])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even) and
    return the 16-bit patterns.  Inputs must be finite."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- routing

def route_uniform(seed: int, T: int, E: int, k: int, exclude=()) -> np.ndarray:
    """k distinct experts per token, uniformly at random, never one in `exclude`."""
    rng = _rng(seed, _TAG_ROUTE)
    keys = rng.random((T, E))
    if len(exclude):
        keys[:, list(exclude)] = 2.0          # sorts after every real key
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def route_zipf(seed: int, T: int, E: int, k: int, s: float = 1.1, n_unused: int = 20) -> np.ndarray:
    """k distinct experts per token drawn without replacement with probability
    proportional to rank^-s, where a seeded permutation assigns the ranks 1..E
    and the last `n_unused` ranks get probability zero (Gumbel top-k)."""
    rng = _rng(seed, _TAG_ROUTE)
    rank = np.empty(E, dtype=np.float64)
    rank[rng.permutation(E)] = np.arange(1, E + 1)
    logp = -s * np.log(rank)
    logp[rank > E - n_unused] = -np.inf
    keys = logp[None, :] + rng.gumbel(size=(T, E))
    return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def route_logits(seed: int, T: int, E: int, k: int):
    """Router logits ~ N(0,1); ids = the k largest (ties to the lower id);
    weights = softmax over all E logits, taken at the chosen ids (not
    renormalised)."""
    rng = _rng(seed, _TAG_ROUTE)
    logits = rng.standard_normal((T, E), dtype=np.float32)
    ids = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    l64 = logits.astype(np.float64)
    p = np.exp(l64 - l64.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    w = np.take_along_axis(p, ids, axis=1).astype(np.float32)
    return ids, w


# ----------------------------------------------------------------------------- tensors

def mxfp4_weights(seed: int, tag: int, E: int, N: int, K: int, exp=(-10, -2)):
    """Uniform nibbles (two per byte) and E8M0 scale bytes 127 + U{exp[0]..exp[1]}."""
    assert K % 32 == 0
    rng = _rng(seed, tag)
    codes = np.frombuffer(rng.bytes(E * N * (K // 2)), dtype=np.uint8).reshape(E, N, K // 2).copy()
    scales = (127 + rng.integers(exp[0], exp[1] + 1, size=(E, N, K // 32))).astype(np.uint8)
    return codes, scales


def e8m0_scales(seed: int, shape, lo: int, hi: int, tag: int = _TAG_SCALES) -> np.ndarray:
    """E8M0 scale bytes drawn uniformly from lo..hi (inclusive), uint8 of `shape`."""
    assert 0 <= lo <= hi <= 255
    return _rng(seed, tag, lo, hi).integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.uint8)


def e4m3_scales(seed: int, shape, lo: int = 0x28, hi: int = 0x48, signs: bool = False) -> np.ndarray:
    """E4M3 scale bytes: the low seven bits uniform in lo..hi (inclusive, at
    most 0x7E so no NaN is drawn), the sign bit random when `signs`."""
    assert 0 <= lo <= hi <= 0x7E
    rng = _rng(seed, _TAG_NV, lo, hi)
    b = rng.integers(lo, hi + 1, size=shape, dtype=np.int64)
    if signs:
        b |= rng.integers(0, 2, size=shape, dtype=np.int64) << 7
    return b.astype(np.uint8)


def tensor_scales(seed: int, E: int) -> np.ndarray:
    """Per-expert float32 scales 2^U{-12..4} * (1 + U{0..7}/8)."""
    rng = _rng(seed, _TAG_NV, E)
    return (np.ldexp(1.0, rng.integers(-12, 5, E)) * (1 + rng.integers(0, 8, E) / 8)).astype(np.float32)


def normal_bf16(seed: int, tag: int, shape) -> np.ndarray:
    rng = _rng(seed, tag)
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def swiglu_shaped_bf16(seed: int, tag: int, shape) -> np.ndarray:
    """Activations distributed like silu(g)*u for independent g, u ~ N(0,1),
    rounded once to bfloat16.  Only the input distribution is drawn here; the
    library's own SwiGLU step is implemented and tested separately."""
    rng = _rng(seed, tag)
    g = rng.standard_normal(shape, dtype=np.float32)
    u = rng.standard_normal(shape, dtype=np.float32)
    return f32_to_bf16_bits(g * u / (np.float32(1) + np.exp(-g)))


def gemm_case(name_or_cfg, seed: int = 0) -> dict:
    """Inputs of one grouped-GEMM workload: routing ids (their per-expert counts
    are the group sizes), sorted activation rows, packed weights."""
    cfg = dict(CONFIGS[name_or_cfg]) if isinstance(name_or_cfg, str) else dict(name_or_cfg)
    E, k, T, K, N = cfg["E"], cfg["k"], cfg["T"], cfg["K"], cfg["N"]
    routing = cfg.get("routing", "uniform")
    if routing == "uniform":
        ids = route_uniform(seed, T, E, k, cfg.get("empty", ()))
    elif routing == "zipf":
        ids = route_zipf(seed, T, E, k)
    else:
        raise ValueError(routing)
    rows = T * k
    if cfg.get("act", "normal") == "swiglu_pairs":
        act = swiglu_shaped_bf16(seed, _TAG_ACT, (rows, K))
    else:
        act = normal_bf16(seed, _TAG_ACT, (rows, K))
    codes, scales = mxfp4_weights(seed, _TAG_W13, E, N, K, cfg.get("exp", (-10, -2)))
    return dict(cfg=cfg, ids=ids, act=act, codes=codes, scales=scales,
                E=E, k=k, T=T, K=K, N=N, rows=rows)


def layer_case(seed: int = 0, T: int | None = None, E: int | None = None,
               hidden: int | None = None, inter: int | None = None, k: int | None = None,
               exp=(-10, -2)) -> dict:
    """Inputs of one MoE layer pass: token activations, router ids and weights,
    w13 (gate|up fused, N = 2*inter) and w2 (N = hidden)."""
    c = CONFIGS["layer"]
    T = c["T"] if T is None else T
    E = c["E"] if E is None else E
    hidden = c["hidden"] if hidden is None else hidden
    inter = c["inter"] if inter is None else inter
    k = c["k"] if k is None else k
    ids, w = route_logits(seed, T, E, k)
    x = normal_bf16(seed, _TAG_X, (T, hidden))
    c13, s13 = mxfp4_weights(seed, _TAG_W13, E, 2 * inter, hidden, exp)
    c2, s2 = mxfp4_weights(seed, _TAG_W2, E, hidden, inter, exp)
    return dict(ids=ids, topk_w=w, x=x, w13_codes=c13, w13_scales=s13, w2_codes=c2, w2_scales=s2,
                T=T, E=E, k=k, hidden=hidden, inter=inter)


def gate_up_f32(seed: int, rows: int, inter: int) -> np.ndarray:
    """Random fused gate|up rows [rows, 2*inter] in float32 for SwiGLU tests."""
    rng = _rng(seed, _TAG_GATE)
    return (rng.standard_normal((rows, 2 * inter), dtype=np.float32) * np.float32(3.0))


def router_weights_uniform(seed: int, T: int, k: int) -> np.ndarray:
    """Positive router weights [T, k] for workloads whose ids are drawn directly
    (uniform or Zipf routing): U(0,1) draws scaled to sum to 1 per token."""
    rng = _rng(seed, _TAG_GATE, 1)
    w = rng.random((T, k)) + 1e-3
    return (w / w.sum(axis=1, keepdims=True)).astype(np.float32)


# name -> (tokens, routing, experts)
WORKLOAD_TOKENS = {"decode_T64": (64, "uniform", 256), "decode_T256": (256, "uniform", 256),
                   "prefill_T4096": (4096, "zipf", 256), "layer_T8192": (8192, "logits", 256),
                   # the layer's band shape (about 192 rows per expert) on 64 experts
                   "layer_E64_T2048": (2048, "logits", 64),
                   # decode-sized bands (one or two rows per expert) on 64 experts
                   "decode_E64_T16": (16, "uniform", 64),
                   # the prefill band mix (half the used experts at 32 rows or fewer) on 96 experts
                   "prefill_E96_T1024": (1024, "zipf", 96)}


def layer_weights(seed: int = 0, E: int = 256, hidden: int = 4096, inter: int = 2048):
    """w13 (gate|up fused, N = 2*inter, K = hidden) and w2 (N = hidden, K =
    inter) codes and scales; the same draws as layer_case/layer_workload with
    the same seed."""
    c13, s13 = mxfp4_weights(seed, _TAG_W13, E, 2 * inter, hidden)
    c2, s2 = mxfp4_weights(seed, _TAG_W2, E, hidden, inter)
    return dict(w13_codes=c13, w13_scales=s13, w2_codes=c2, w2_scales=s2)


def workload_tokens(name: str, seed: int = 0, k: int = 6, hidden: int = 4096) -> dict:
    """Routing ids, router weights and token activations of a named full-path
    workload (no weights): the draws layer_workload makes for the same name
    and seed."""
    T, routing, E = WORKLOAD_TOKENS[name]
    if routing == "logits":
        ids, w = route_logits(seed, T, E, k)
    else:
        ids = route_uniform(seed, T, E, k) if routing == "uniform" else route_zipf(seed, T, E, k)
        w = router_weights_uniform(seed, T, k)
    x = normal_bf16(seed, _TAG_X, (T, hidden))
    return dict(ids=ids, topk_w=w, x=x, T=T, E=E, k=k, hidden=hidden)


def layer_workload(name: str, seed: int = 0) -> dict:
    """Full-path inputs (route sort -> w13 -> SwiGLU -> w2 -> combine) for the
    named workload; the token count and routing follow the named config."""
    E, k, hidden, inter = 256, 6, 4096, 2048
    if name == "layer_T8192":
        return layer_case(seed)
    T, routing = {"decode_T64": (64, "uniform"), "decode_T256": (256, "uniform"),
                  "prefill_T4096": (4096, "zipf")}[name]
    ids = route_uniform(seed, T, E, k) if routing == "uniform" else route_zipf(seed, T, E, k)
    x = normal_bf16(seed, _TAG_X, (T, hidden))
    c13, s13 = mxfp4_weights(seed, _TAG_W13, E, 2 * inter, hidden)
    c2, s2 = mxfp4_weights(seed, _TAG_W2, E, hidden, inter)
    return dict(ids=ids, topk_w=router_weights_uniform(seed, T, k), x=x, w13_codes=c13,
                w13_scales=s13, w2_codes=c2, w2_scales=s2, T=T, E=E, k=k, hidden=hidden, inter=inter)
