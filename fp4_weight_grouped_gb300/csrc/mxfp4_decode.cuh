// Exact decode of MXFP4 weights to bfloat16: e2m1 code times 2^(s - 127).
//
// "Running DeepSeek V4 Flash on TPU v6", section 1: the eight e2m1 magnitudes are
// 0, 0.5, 1, 1.5, 2, 3, 4, 6, and the per-32 block scale is applied to the decoded
// values before the matmul.  Every such product with s in 0..252 is a bf16 number
// (normal or subnormal), so the decode is exact.  Code 0x8 (-0) yields +0
// ("DeepSeek-V4-Flash-0731-NVFP4", the E2M1 -0 -> +0 canonicalisation).
//
// GB300 design.  Integer logic (LOP3/PRMT/shifts) issues at half rate on the SM's
// ALU pipe, while IMAD and bf16x2 FMA go to the FMA pipe, so the decode splits
// its work across both:
//   1. Two codes of one 32-bit code word, nibbles j and j+4, are masked into the
//      low nibble of each 16-bit half (one LOP3).
//   2. One IMAD by 0x1040 copies each nibble to bits 6..9 and 12..15 of its half;
//      a second LOP3 keeps bits 6..8 (exponent+mantissa e1 e0 m) and bit 15
//      (sign).  As a bf16 pattern that is exactly e2m1 * 2^-126: e = 0 lands in
//      bf16's subnormal range, which represents 0 and 0.5 * 2^-126 exactly.
//   3. One fma.rn.bf16x2 by 2^(s-1) (and +0) gives e2m1 * 2^(s-127) exactly; the
//      +0 addend turns the -0 of code 0x8 into +0.  For s > 128 the constant
//      would overflow, so the product is split into * 2^126 then * 2^(s-127).
// So one pair of weights costs 2 ALU + 2 FMA-pipe instructions.
//
// Pairing nibbles j and j+4 means one 32-bit result holds elements (8w + j,
// 8w + j + 4) of a code word w.  The GEMM therefore consumes the reduction
// dimension in the order [0,4,1,5,2,6,3,7] within every group of 8, and the
// activations must use the same order (the "K8-interleaved" layout).
#pragma once

#include "device_common.cuh"

namespace moe {

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// bf16 patterns of e2m1 * 2^-126 for the code pairs of word c:
// x[j] = (code j, code j+4), j = 0..3.
__device__ __forceinline__ void e2m1_pairs_scaled_down(uint32_t c, uint32_t (&x)[4]) {
    const uint32_t c8 = c >> 8;
    x[0] = ((c & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;
    x[1] = ((c & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;
    x[2] = ((c8 & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;
    x[3] = ((c8 & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;
}

// bf16x2 of 2^(s-1) in both halves, for scale byte s in 0..128.
__device__ __forceinline__ uint32_t scale_pair_single(uint32_t s) {
    return s * 0x00800080u + 0x3F003F00u;          // (s + 126) << 7, twice
}

// Scale pairs (first, second) for any s in 0..252: s <= 128 -> (2^(s-1), 1);
// s > 128 -> (2^126, 2^(s-127)).
__device__ __forceinline__ void scale_pair_split(uint32_t s, uint32_t &first, uint32_t &second) {
    const bool big = s > 128u;
    first = big ? 0x7E807E80u : scale_pair_single(s);
    second = big ? s * 0x00800080u : 0x3F803F80u;
}

// Decode one 32-code block (16 bytes in c[0..3]) into 16 bf16 pairs in GEMM
// reduction order; o[4w + j] = (element 8w + j, element 8w + j + 4).
__device__ __forceinline__ void decode32_single(const uint32_t (&c)[4], uint32_t S,
                                                uint32_t *o) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t x[4];
        e2m1_pairs_scaled_down(c[w], x);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[4 * w + j] = bf16x2_fma(x[j], S, 0u);
    }
}

__device__ __forceinline__ void decode32_split(const uint32_t (&c)[4], uint32_t S1, uint32_t S2,
                                               uint32_t *o) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t x[4];
        e2m1_pairs_scaled_down(c[w], x);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[4 * w + j] = bf16x2_fma(bf16x2_fma(x[j], S1, 0u), S2, 0u);
    }
}

// Any scale byte: 0..252 decode exactly; 253..255 give NaN and return false.
__device__ __forceinline__ bool decode32_any(const uint32_t (&c)[4], uint32_t s, uint32_t *o) {
    if (s > 252u) {
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = 0x7FC07FC0u;
        return false;
    }
    uint32_t S1, S2;
    scale_pair_split(s, S1, S2);
    decode32_split(c, S1, S2, o);
    return true;
}

// K8 interleave of 8 bf16 (one 16-byte chunk): natural (e0..e7) in (x, y, z, w)
// -> (e0,e4), (e1,e5), (e2,e6), (e3,e7).
__device__ __forceinline__ uint4 interleave8(uint4 v) {
    uint4 r;
    r.x = prmt(v.x, v.z, 0x5410u);
    r.y = prmt(v.x, v.z, 0x7632u);
    r.z = prmt(v.y, v.w, 0x5410u);
    r.w = prmt(v.y, v.w, 0x7632u);
    return r;
}

// Inverse of interleave8.
__device__ __forceinline__ uint4 deinterleave8(uint4 v) {
    uint4 r;
    r.x = prmt(v.x, v.y, 0x5410u);
    r.y = prmt(v.z, v.w, 0x5410u);
    r.z = prmt(v.x, v.y, 0x7632u);
    r.w = prmt(v.z, v.w, 0x7632u);
    return r;
}

}  // namespace moe
