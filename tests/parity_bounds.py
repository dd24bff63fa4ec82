"""Tolerance of SwiGLU computed from GEMM sums that carry the GEMM tolerance
(the fused w13 + SwiGLU epilogue), against the oracle's SwiGLU of the oracle's
fp64 gate/up sums.

With g, u the exact sums, t_g, t_u their GEMM tolerances (1e-5 * sum|a w| +
1e-6) and g', u' the kernel's f32 sums (|g' - g| <= t_g, |u' - u| <= t_u):
  |silu(g') u' - silu(g) u| <= max|silu'| t_g (|u| + t_u) + |silu(g)| t_u,
  max over x of silu'(x) = sigma(x) (1 + x (1 - sigma(x))) < 1.0998,
plus the final rounding to bf16 and the oracle's own rounding to bf16 (one
bf16 ulp each, counted as two ulps of the oracle's value).
"""
import numpy as np

SILU_SLOPE_MAX = 1.1


def bf16_ulp(x):
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    return np.ldexp(1.0, (np.maximum(e, -126) - 7).astype(np.int64))


def bf16_bits_to_f64(bits):
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def swiglu_from_gemm_bound(y13_ref, mag13, h_ref_bits, rel=1e-5, abs_=1e-6):
    """Per-element bound for h given the oracle's fp64 gate/up sums y13_ref
    [rows, 2I], their sum|a w| mag13, and the oracle's bf16 SwiGLU h_ref_bits."""
    I = y13_ref.shape[1] // 2
    g, u = y13_ref[:, :I], y13_ref[:, I:]
    tg, tu = rel * mag13[:, :I] + abs_, rel * mag13[:, I:] + abs_
    silu_g = np.abs(g) / (1.0 + np.exp(-np.clip(g, -700, 700)))
    h_ref = bf16_bits_to_f64(h_ref_bits)
    return 2.0 * bf16_ulp(h_ref) + SILU_SLOPE_MAX * tg * (np.abs(u) + tu) + silu_g * tu


def check_swiglu_from_gemm(h_bits, y13_ref, mag13, h_ref_bits, what=""):
    bound = swiglu_from_gemm_bound(y13_ref, mag13, h_ref_bits)
    diff = np.abs(bf16_bits_to_f64(h_bits) - bf16_bits_to_f64(h_ref_bits))
    bad = ~(diff <= bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {diff.size} outside the SwiGLU bound; "
                           f"worst ratio {float(np.max(diff / bound)):.3g}")
