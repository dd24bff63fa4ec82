// Exact decode of MXFP4 weights to bfloat16: e2m1 code times 2^(s - 127).
//
// "Running DeepSeek V4 Flash on TPU v6", section 1: the eight e2m1 magnitudes are
// 0, 0.5, 1, 1.5, 2, 3, 4, 6, and the per-32 block scale is applied to the decoded
// values before the matmul.  Every such product with s in 0..252 is a bf16 number,
// so the decode is exact.  Code 0x8 (-0) yields +0 ("DeepSeek-V4-Flash-0731-NVFP4",
// the E2M1 -0 -> +0 canonicalisation).
//
// GB300 design: instead of the page's three vector ops on a re-encoded integer,
// each 32-code block gets a byte lookup table for its scale s.  For s in 2..252
// every bf16 result is a normal number whose 16-bit pattern is
//     V[m] = (s-1)<<7 + {0, 0, 0x80, 0xC0, 0x100, 0x140, 0x180, 0x1C0}[m]   (m >= 1),
//     V[0] = 0,
// for magnitude index m = 2e + mant.  The low and high bytes of V[0..7] form two
// 8-byte tables; `prmt` looks four nibbles up at once, the sign bit (of nonzero
// codes only) is OR-ed into the high byte, and a final `prmt` interleaves the
// bytes into bf16 pairs.  Scale bytes 0 and 1 give bf16 subnormals and take a
// slower exact path; 253..255 are out of range (status MOE_ERR_DATA, NaN).
#pragma once

#include "device_common.cuh"

namespace moe {

struct DecodeLut {
    uint32_t lo0, lo1, hi0, hi1;   // bytes 0..7: low / high byte of V[m]
};

// Lookup table for scale byte s (valid for 2 <= s <= 252; zeros otherwise).
__device__ __forceinline__ DecodeLut make_decode_lut(uint32_t s) {
    DecodeLut t = {0u, 0u, 0u, 0u};
    if (s >= 2u && s <= 252u) {
        const uint32_t q = (s - 1u) << 7;          // bf16 bits of 0.5 * 2^(s-127)
        const uint32_t qq = q * 0x10001u;
        const uint32_t v01 = q << 16;              // V0 = 0,        V1 = 0.5
        const uint32_t v23 = qq + 0x00C00080u;     // V2 = 1.0,      V3 = 1.5
        const uint32_t v45 = qq + 0x01400100u;     // V4 = 2.0,      V5 = 3.0
        const uint32_t v67 = qq + 0x01C00180u;     // V6 = 4.0,      V7 = 6.0
        t.lo0 = prmt(v01, v23, 0x6420u);
        t.lo1 = prmt(v45, v67, 0x6420u);
        t.hi0 = prmt(v01, v23, 0x7531u);
        t.hi1 = prmt(v45, v67, 0x7531u);
    }
    return t;
}

// Eight codes (one 32-bit word, code i in bits 4i..4i+3, element order) to four
// bf16 pairs (element 2j in the low half of o[j]).
__device__ __forceinline__ void decode8_lut(uint32_t c, const DecodeLut &t, uint32_t *o) {
    const uint32_t m = c & 0x77777777u;                       // magnitude index per nibble
    const uint32_t sgn = (m + 0x77777777u) & c & 0x88888888u; // sign bit of nonzero codes
    const uint32_t mh = m >> 16;
    uint32_t L0 = prmt(t.lo0, t.lo1, m);                      // low bytes, codes 0..3
    uint32_t H0 = prmt(t.hi0, t.hi1, m);                      // high bytes, codes 0..3
    uint32_t L1 = prmt(t.lo0, t.lo1, mh);                     // codes 4..7
    uint32_t H1 = prmt(t.hi0, t.hi1, mh);
    const uint32_t s4 = sgn << 4;                             // even-code signs to bit 7 of a byte
    H0 |= prmt(s4, sgn, 0x5140u) & 0x80808080u;
    H1 |= prmt(s4, sgn, 0x7362u) & 0x80808080u;
    o[0] = prmt(L0, H0, 0x5140u);
    o[1] = prmt(L0, H0, 0x7362u);
    o[2] = prmt(L1, H1, 0x5140u);
    o[3] = prmt(L1, H1, 0x7362u);
}

// Exact slow path for one code with scale byte 0 or 1 (bf16 subnormal range).
__device__ __forceinline__ uint32_t decode1_small_scale(uint32_t code, uint32_t s) {
    const uint32_t mag = code & 7u;
    const uint32_t e = mag >> 1, mt = mag & 1u;
    // e2m1 magnitude as f32 bits: e == 0 -> 0 or 0.5; else 2^(e-1) * (1 + mt/2).
    uint32_t fbits;
    if (mag == 0u) fbits = 0u;
    else if (e == 0u) fbits = 0x3F000000u;                      // 0.5
    else fbits = ((126u + e) << 23) | (mt << 22);
    const float v = __uint_as_float(fbits);
    const float scale = __uint_as_float(s == 0u ? 0x00400000u : 0x00800000u);  // 2^-127, 2^-126
    float w = v * scale;                                        // exact (no flush to zero)
    uint32_t b = __float_as_uint(w) >> 16;                      // exact: at most 2 significant bits
    if ((code & 8u) && mag) b |= 0x8000u;
    return b;
}

// Decode one 32-code block (16 bytes in c[0..3]) with scale byte s into 16 bf16
// pairs.  `lut` must be make_decode_lut(s).  Returns false if s > 252 (the block
// is then filled with NaN).
__device__ __forceinline__ bool decode32(const uint32_t (&c)[4], uint32_t s, const DecodeLut &lut,
                                         uint32_t (&o)[16]) {
    if (s - 2u <= 250u) {
#pragma unroll
        for (int i = 0; i < 4; ++i) decode8_lut(c[i], lut, &o[4 * i]);
        return true;
    }
    if (s <= 1u) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t b = (c[i] >> (8 * j)) & 0xFFu;
                o[4 * i + j] = decode1_small_scale(b & 15u, s) |
                               (decode1_small_scale(b >> 4, s) << 16);
            }
        return true;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = 0x7FC07FC0u;
    return false;
}

}  // namespace moe
