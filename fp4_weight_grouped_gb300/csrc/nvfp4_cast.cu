// Lossless cast of MXFP4 expert scales to NVFP4's two-level scaling
// ("DeepSeek-V4-Flash-0731-NVFP4", "The lossless weight cast").
//
// Per expert e (its whole [N, K/32] E8M0 scale tensor, so the rows of a fused
// w1/w3 tensor share one value), with m = the largest scale byte:
//   weight_scale_2[e] = 2^(m - 127 - 8), an exact f32 (subnormal below 2^-126);
//   both per-16 E4M3 scales of 32-block b = 2^(s_b - m + 8), exact for
//   exponents -9..8 (E4M3 normals 2^-6..2^8, subnormals 2^-7..2^-9);
// so per-16 scale x per-tensor scale = 2^(s_b - 127), the MXFP4 block scale,
// and the unchanged e2m1 codes dequantize to identical values.  A block with
// s_b < m - 17 has no exact E4M3 scale: it is written as 0 and counted.
//
// Every E4M3 byte depends on the expert's maximum, so the data is read, reduced
// across the expert, then converted.  Two forms:
//   * one pass (the usual shapes): one thread-block cluster of up to 16 CTAs
//     of 128 threads per expert.  Every thread loads its 256 scale bytes into
//     registers (16 loads of 16 bytes in flight), the CTAs of the cluster
//     exchange their maxima through distributed shared memory, and each thread
//     converts from its registers and stores.  The scales are read from HBM
//     once: 3 bytes of traffic per scale byte, the algorithmic minimum.
//   * two passes (an expert over 512 KiB, or buffers off 16-byte boundaries):
//     a per-expert maximum into scratch, then the conversion.
// Four scale bytes are converted at a time with byte-parallel integer
// arithmetic in one 32-bit register (below, convert_word).  Results are
// integers, identical from run to run.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "launch.h"

namespace moe {
namespace cast {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kBlocksPerSM = 8;            // two-pass grid: blocks per SM
constexpr long long kMinChunk = 4096;      // two-pass grid: smallest chunk
constexpr int kRegVec = 16;                // one pass: 16-byte words per thread
// One pass: threads per CTA.  A CTA holds 32 KiB in registers and a cluster of
// up to 16 CTAs (non-portable size, opted in) covers an expert's 512 KiB;
// four or five CTAs fit an SM, so one expert's stores overlap another's loads.
constexpr int kOneNT = 128;
constexpr long long kSlice = static_cast<long long>(kOneNT) * kRegVec * 16;
constexpr int kMaxCluster = kOneNT == 256 ? 8 : 16;
constexpr uint32_t kOnes = 0x01010101u, kHigh = 0x80808080u;

__device__ __forceinline__ uint32_t max_byte4(uint32_t w) {
    return max(max(w & 0xFFu, (w >> 8) & 0xFFu), max((w >> 16) & 0xFFu, w >> 24));
}

__device__ __forceinline__ uint32_t max_byte16(uint32_t acc, uint4 w) {
    return __vmaxu4(acc, __vmaxu4(__vmaxu4(w.x, w.y), __vmaxu4(w.z, w.w)));
}

// E4M3 byte of 2^p for p <= 8: normal for p >= -6 (biased exponent p + 7,
// mantissa 0), subnormal 2^-7..2^-9 (mantissa 4, 2, 1), 0 below 2^-9.
__device__ __forceinline__ uint32_t e4m3_pow2(int p) {
    if (p >= -6) return static_cast<uint32_t>(p + 7) << 3;
    if (p >= -9) return 1u << (p + 9);
    return 0u;
}

// Four scale bytes of one expert -> their four E4M3 bytes, byte-parallel in
// one register.  M = the expert's maximum in all four bytes; every byte of w is
// at most that maximum, so M - w subtracts byte by byte without borrows.  With
// d = m - s per byte the result is e4m3_pow2(8 - d):
//   g = 18 - d clamped at 0 (d >= 128 and d > 18 give 0);
//   g >= 4:  normal, biased exponent g - 3, byte (g - 3) << 3;
//   g = 1, 2, 3: subnormal 1, 2, 4 (g plus one when g = 3);  g = 0: 0.
// `in_range` counts the bytes with g >= 1 (p >= -9).  Every intermediate
// byte stays below 256, so no carry crosses into a neighbouring byte.
__device__ __forceinline__ uint32_t convert_word(uint32_t w, uint32_t M, uint32_t &in_range) {
    const uint32_t d = M - w;
    const uint32_t x = (0x12u * kOnes | kHigh) - (d & 0x7F7F7F7Fu);     // 146 - (d & 127) >= 19
    const uint32_t ok = x & ~d & kHigh;                                  // d <= 18
    const uint32_t g = x & (ok - (ok >> 7)) & 0x1F1F1F1Fu;               // 18 - d, or 0
    in_range += __popc((g + 0x7F7F7F7Fu) & kHigh);                       // g >= 1
    const uint32_t y = (g | kHigh) - 4u * kOnes;                         // bit 7: g >= 4
    const uint32_t nh = y & kHigh;
    const uint32_t nmask = nh - (nh >> 7);                               // 0x7F where normal
    const uint32_t normal = (y & 0x0F0F0F0Fu) * 8u + 8u * kOnes;         // (g - 3) << 3 there
    const uint32_t sub = g + ((g >> 1) & g & kOnes);                     // 1, 2, 4 for g = 1, 2, 3
    return (normal & nmask) | (sub & ~nmask);
}

// 16 scale bytes -> 32 output bytes: every E4M3 byte twice (the two 16-element
// halves of its 32-block), in block order.
__device__ __forceinline__ void convert16(uint4 w, uint32_t M, uint32_t &in_range, uint4 &o0,
                                          uint4 &o1) {
    const uint32_t a = convert_word(w.x, M, in_range), b = convert_word(w.y, M, in_range);
    const uint32_t c = convert_word(w.z, M, in_range), d = convert_word(w.w, M, in_range);
    o0 = make_uint4(prmt(a, 0u, 0x1100u), prmt(a, 0u, 0x3322u), prmt(b, 0u, 0x1100u),
                    prmt(b, 0u, 0x3322u));
    o1 = make_uint4(prmt(c, 0u, 0x1100u), prmt(c, 0u, 0x3322u), prmt(d, 0u, 0x1100u),
                    prmt(d, 0u, 0x3322u));
}

// 2^(m - 135) as f32 bits; m >= 0 keeps the exponent >= -135 (a subnormal).
__device__ __forceinline__ float weight_scale_2_of(uint32_t m) {
    const int x = static_cast<int>(m) - 135;
    return __uint_as_float(x >= -126 ? static_cast<uint32_t>(x + 127) << 23 : 1u << (x + 149));
}

// Every thread gets op over the block's per-warp values v (each warp passes
// one warp-uniform value).  Callers separate two uses of warp_vals by a barrier.
template <int NT, typename T, typename Op>
__device__ __forceinline__ T block_reduce(T v, Op op, T *warp_vals) {
    if ((threadIdx.x & 31) == 0) warp_vals[threadIdx.x >> 5] = v;
    __syncthreads();
    T r = warp_vals[0];
    for (int w = 1; w < NT / 32; ++w) r = op(r, warp_vals[w]);
    return r;
}

// ------------------------------------------------------------------ one pass

// Grid (C, E) with clusters of (C, 1, 1): cluster e converts expert e; CTA c
// holds bytes [c * kSlice, min((c + 1) * kSlice, per_expert)) in registers.
// Needs per_expert % 16 == 0, per_expert <= C * kSlice, 16-byte aligned bases.
__global__ void __launch_bounds__(kOneNT, kOneNT == 256 ? 2 : 4)
onepass_kernel(const uint8_t *__restrict__ scales, long long per_expert, uint8_t *__restrict__ e4m3,
               float *__restrict__ weight_scale_2, unsigned long long *__restrict__ out_of_range,
               int *status) {
    cg::cluster_group cluster = cg::this_cluster();
    const int e = blockIdx.y;
    const unsigned rank = cluster.block_rank();
    const unsigned csize = cluster.num_blocks();
    __shared__ uint32_t expert_max, expert_in_range;   // gathered from the whole cluster
    __shared__ uint32_t warp_vals[kOneNT / 32];
    if (threadIdx.x == 0) {
        expert_max = 0;
        expert_in_range = 0;
    }
    // Arrive now, wait after the loads: the peers' maxima are written into this
    // CTA's expert_max only once every CTA of the cluster has started and
    // initialised it, and the barrier's latency hides behind the loads.

    const long long lo = static_cast<long long>(rank) * kSlice;
    const long long nvec = max(0LL, min(kSlice, per_expert - lo)) / 16;
    const uint4 *src = reinterpret_cast<const uint4 *>(scales + static_cast<long long>(e) * per_expert + lo);
    uint4 w[kRegVec];
#pragma unroll
    for (int u = 0; u < kRegVec; ++u) {
        const long long j = threadIdx.x + static_cast<long long>(u) * kOneNT;
        w[u] = j < nvec ? __ldcs(src + j) : make_uint4(0, 0, 0, 0);
    }
    uint32_t acc = 0;
#pragma unroll
    for (int u = 0; u < kRegVec; ++u) acc = max_byte16(acc, w[u]);
    const uint32_t m_warp = __reduce_max_sync(0xffffffffu, max_byte4(acc));
    const uint32_t m_cta =
        block_reduce<kOneNT>(m_warp, [](uint32_t a, uint32_t b) { return max(a, b); }, warp_vals);
    cluster.sync();                                 // every CTA's expert_max is initialised
    if (threadIdx.x < csize) atomicMax(cluster.map_shared_rank(&expert_max, threadIdx.x), m_cta);
    cluster.sync();                                 // every CTA's maximum has arrived everywhere;
                                                    // no shared memory of a peer is used after this
    const uint32_t m = expert_max;
    const uint32_t M = m * kOnes;
    uint4 *dst = reinterpret_cast<uint4 *>(e4m3 + 2 * (static_cast<long long>(e) * per_expert + lo));
    uint32_t in_range = 0;
#pragma unroll
    for (int u = 0; u < kRegVec; ++u) {
        const long long j = threadIdx.x + static_cast<long long>(u) * kOneNT;
        if (j < nvec) {
            uint4 o0, o1;
            convert16(w[u], M, in_range, o0, o1);
            __stcs(dst + 2 * j, o0);
            __stcs(dst + 2 * j + 1, o1);
        }
    }
    const uint32_t r_warp = __reduce_add_sync(0xffffffffu, in_range);
    __syncthreads();                                // warp_vals reused
    const uint32_t r_cta =
        block_reduce<kOneNT>(r_warp, [](uint32_t a, uint32_t b) { return a + b; }, warp_vals);
    if (threadIdx.x == 0) atomicAdd(cluster.map_shared_rank(&expert_in_range, 0), r_cta);
    cluster.sync();                                 // all counts are in CTA 0
    if (rank == 0 && threadIdx.x == 0) {
        out_of_range[e] = static_cast<unsigned long long>(per_expert) - expert_in_range;
        weight_scale_2[e] = weight_scale_2_of(m);
        if (m == 255u) set_status(status, MOE_ERR_DATA);
    }
}

// ---------------------------------------------------------------- two passes

// Bytes [lo, hi) of expert e's scale tensor for block (x, e).
struct Span {
    long long lo, hi;
};
__device__ __forceinline__ Span block_span(long long per_expert, long long chunk) {
    const long long lo = static_cast<long long>(blockIdx.x) * chunk;
    return {lo, min(lo + chunk, per_expert)};
}

__device__ __forceinline__ long long head_bytes(const uint8_t *p, const Span &sp) {
    return min(static_cast<long long>((16 - (reinterpret_cast<uintptr_t>(p + sp.lo) & 15)) & 15),
               sp.hi - sp.lo);
}

// Pass 1: largest scale byte of each expert; 255 (the E8M0 NaN) records MOE_ERR_DATA.
__global__ void __launch_bounds__(kThreads)
kmax_kernel(const uint8_t *__restrict__ scales, long long per_expert, long long chunk,
            int *__restrict__ kmax, int *status) {
    const int e = blockIdx.y;
    const uint8_t *base = scales + static_cast<long long>(e) * per_expert;
    const Span sp = block_span(per_expert, chunk);
    // Single bytes up to the first 16-byte boundary, 16-byte loads, single-byte tail.
    const long long head = head_bytes(base, sp);
    uint32_t acc = 0;
    for (long long i = sp.lo + threadIdx.x; i < sp.lo + head; i += kThreads) acc = max(acc, uint32_t(base[i]));
    const long long vlo = sp.lo + head;
    const long long nvec = (sp.hi - vlo) / 16;
    const uint4 *v = reinterpret_cast<const uint4 *>(base + vlo);
    for (long long i = threadIdx.x; i < nvec; i += 4 * kThreads) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long long j = i + u * kThreads;
            w[u] = j < nvec ? __ldg(v + j) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) acc = max_byte16(acc, w[u]);
    }
    for (long long i = vlo + nvec * 16 + threadIdx.x; i < sp.hi; i += kThreads) acc = max(acc, uint32_t(base[i]));
    __shared__ uint32_t warp_vals[kThreads / 32];
    const uint32_t m_warp = __reduce_max_sync(0xffffffffu, max_byte4(acc));
    const uint32_t m = block_reduce<kThreads>(m_warp, [](uint32_t a, uint32_t b) { return max(a, b); }, warp_vals);
    if (threadIdx.x == 0) {
        atomicMax(&kmax[e], static_cast<int>(m));
        if (m == 255u) set_status(status, MOE_ERR_DATA);
    }
}

__device__ __forceinline__ void convert1(const uint8_t *src, uint8_t *dst, long long i, int m,
                                         uint32_t &in_range) {
    const int p = static_cast<int>(src[i]) - m + 8;
    in_range += p >= -9 ? 1u : 0u;
    const uint8_t v = static_cast<uint8_t>(e4m3_pow2(p));
    dst[2 * i] = v;
    dst[2 * i + 1] = v;
}

// Pass 2: per-16 scales of expert e, its per-tensor scale and out-of-range count.
__global__ void __launch_bounds__(kThreads)
convert_kernel(const uint8_t *__restrict__ scales, long long per_expert, long long chunk,
               const int *__restrict__ kmax, uint8_t *__restrict__ e4m3,
               float *__restrict__ weight_scale_2, unsigned long long *__restrict__ out_of_range) {
    const int e = blockIdx.y;
    const int m = kmax[e];
    const uint32_t M = static_cast<uint32_t>(m) * kOnes;
    const uint8_t *src = scales + static_cast<long long>(e) * per_expert;
    uint8_t *dst = e4m3 + 2 * static_cast<long long>(e) * per_expert;
    const Span sp = block_span(per_expert, chunk);
    uint32_t in_range = 0;
    const long long head = head_bytes(src, sp);
    const long long vlo = sp.lo + head;
    // The vector path needs the output of byte vlo on a 16-byte boundary too.
    const bool vec = (reinterpret_cast<uintptr_t>(dst + 2 * vlo) & 15) == 0;
    const long long nvec = vec ? (sp.hi - vlo) / 16 : 0;
    for (long long i = sp.lo + threadIdx.x; i < sp.lo + head; i += kThreads) convert1(src, dst, i, m, in_range);
    const uint4 *v = reinterpret_cast<const uint4 *>(src + vlo);
    uint4 *o = reinterpret_cast<uint4 *>(dst + 2 * vlo);
    for (long long i = threadIdx.x; i < nvec; i += 2 * kThreads) {
        uint4 w[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const long long j = i + u * kThreads;
            w[u] = j < nvec ? __ldcs(v + j) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const long long j = i + u * kThreads;
            if (j < nvec) {
                uint4 o0, o1;
                convert16(w[u], M, in_range, o0, o1);
                __stcs(o + 2 * j, o0);
                __stcs(o + 2 * j + 1, o1);
            }
        }
    }
    for (long long i = vlo + nvec * 16 + threadIdx.x; i < sp.hi; i += kThreads) convert1(src, dst, i, m, in_range);
    __shared__ uint32_t warp_vals[kThreads / 32];
    const uint32_t r_warp = __reduce_add_sync(0xffffffffu, in_range);
    const uint32_t r = block_reduce<kThreads>(r_warp, [](uint32_t a, uint32_t b) { return a + b; }, warp_vals);
    if (threadIdx.x == 0) {
        const unsigned long long bad = static_cast<unsigned long long>(sp.hi - sp.lo) - r;
        if (bad) atomicAdd(&out_of_range[e], bad);
        if (blockIdx.x == 0) weight_scale_2[e] = weight_scale_2_of(static_cast<uint32_t>(m));
    }
}

}  // namespace cast

bool nvfp4_cast_one_pass(const void *scales, const void *e4m3, int N, int K) {
    const long long per_expert = static_cast<long long>(N) * (K / 32);
    return per_expert % 16 == 0 && per_expert <= cast::kMaxCluster * cast::kSlice &&
           (reinterpret_cast<uintptr_t>(scales) & 15) == 0 && (reinterpret_cast<uintptr_t>(e4m3) & 15) == 0;
}

moe_status launch_mxfp4_to_nvfp4(const uint8_t *scales, int E, int N, int K, uint8_t *e4m3,
                                 float *weight_scale_2, unsigned long long *out_of_range,
                                 int *kmax_scratch, int *status, cudaStream_t stream, int num_sms,
                                 int *launches) {
    using namespace cast;
    *launches = 0;
    const long long per_expert = static_cast<long long>(N) * (K / 32);
    if (nvfp4_cast_one_pass(scales, e4m3, N, K)) {
        const unsigned csize = static_cast<unsigned>((per_expert + kSlice - 1) / kSlice);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(csize, static_cast<unsigned>(E), 1);
        cfg.blockDim = dim3(kOneNT, 1, 1);
        if (kMaxCluster > 8) {
            // Clusters beyond the portable 8 need the opt-in (set once per process).
            static const cudaError_t opt = cudaFuncSetAttribute(
                onepass_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (opt != cudaSuccess) return MOE_ERR_CUDA;
        }
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = csize;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, onepass_kernel, scales, per_expert, e4m3, weight_scale_2,
                               out_of_range, status) != cudaSuccess)
            return MOE_ERR_CUDA;
        *launches = 1;
        return MOE_OK;
    }
    if (cudaMemsetAsync(kmax_scratch, 0, static_cast<size_t>(E) * sizeof(int), stream) != cudaSuccess ||
        cudaMemsetAsync(out_of_range, 0, static_cast<size_t>(E) * sizeof(unsigned long long), stream) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    // Split every expert into gx equal chunks (multiples of 16 bytes) so that
    // the grid holds about kBlocksPerSM blocks per SM.
    const long long target = static_cast<long long>(kBlocksPerSM) * num_sms;
    long long gx = (target + E - 1) / E;
    long long chunk = (per_expert + gx - 1) / gx;
    chunk = max(kMinChunk, (chunk + 15) & ~15LL);
    gx = (per_expert + chunk - 1) / chunk;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(E));
    kmax_kernel<<<grid, kThreads, 0, stream>>>(scales, per_expert, chunk, kmax_scratch, status);
    convert_kernel<<<grid, kThreads, 0, stream>>>(scales, per_expert, chunk, kmax_scratch, e4m3,
                                                  weight_scale_2, out_of_range);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    *launches = 2;
    return MOE_OK;
}

}  // namespace moe
