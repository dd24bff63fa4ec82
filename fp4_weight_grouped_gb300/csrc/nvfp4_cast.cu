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
//   * one pass (the usual shapes): persistent thread-block clusters of C <= 8
//     CTAs, each CTA owning one 64 KiB slice of an expert's scales, cluster c
//     converting experts c, c + #clusters, ...  A slice arrives by bulk copy
//     (cp.async.bulk) into shared memory, every thread moves its 256 bytes into
//     registers, and the copy of the cluster's next expert starts at once, so it
//     overlaps this expert's conversion and stores.  The CTAs of the cluster
//     exchange their maxima (and the in-range counts of the previous expert) by
//     asynchronous stores into each peer's shared memory that complete on the
//     peer's mbarrier: no cluster barrier inside the loop, whose release would
//     make every thread wait for its output stores.  The scales are read from
//     HBM once: 3 bytes of traffic per scale byte, the algorithmic minimum.
//   * two passes (an expert over 512 KiB, or buffers off 16-byte boundaries):
//     a per-expert maximum into scratch, then the conversion.
// Four scale bytes are converted at a time with byte-parallel integer
// arithmetic in one 32-bit register (below, convert_word).  Results are
// integers, identical from run to run.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "device_common.cuh"
#include "launch.h"

namespace moe {
namespace cast {

constexpr int kThreads = 256;
constexpr int kBlocksPerSM = 8;            // two-pass grid: blocks per SM
constexpr long long kMinChunk = 4096;      // two-pass grid: smallest chunk
// One pass: 256 threads per CTA, 32 eight-byte words each: a 64 KiB slice per
// CTA, two CTAs per SM, clusters of up to 8 CTAs (512 KiB per expert).
constexpr int kOneNT = 256;
constexpr int kOneWords = 32;
constexpr long long kSlice = static_cast<long long>(kOneNT) * kOneWords * 8;
constexpr int kMaxCluster = 8;
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

// Shared memory of the one-pass kernel.
struct OnePassSmem {
    uint8_t slice[kSlice];                 // this CTA's slice of the current expert
    uint64_t full[2];                      // bulk copy of use k: full[k & 1], parity (k >> 1) & 1
    uint64_t xfull[2];                     // exchange of use k: the same scheme
    uint32_t xch[2][kMaxCluster][2];       // (maximum, in-range count) from each CTA
    uint32_t wmax[kOneNT / 32], wcnt[kOneNT / 32];
};

// Grid (C * clusters) with clusters of (C, 1, 1), C = ceil(per_expert / kSlice):
// CTA rank r holds bytes [r * kSlice, min((r + 1) * kSlice, per_expert)) of
// every expert its cluster converts.  Needs per_expert % 16 == 0, 16-byte
// aligned bases.
__global__ void __launch_bounds__(kOneNT, 2)
onepass_kernel(const uint8_t *__restrict__ scales, long long per_expert, int E, uint8_t *__restrict__ e4m3,
               float *__restrict__ weight_scale_2, unsigned long long *__restrict__ out_of_range,
               int *status, uint64_t limit_ns) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    OnePassSmem &sm = *reinterpret_cast<OnePassSmem *>(smem_raw);
    uint32_t C;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(C));
    const uint32_t rank = cluster_rank();
    const int n_clusters = static_cast<int>(gridDim.x / C);
    const int first = static_cast<int>(blockIdx.x / C);
    const int tid = threadIdx.x;
    const long long lo = static_cast<long long>(rank) * kSlice;
    const uint32_t len = static_cast<uint32_t>(max(0LL, min(kSlice, per_expert - lo)));
    const int nwords = static_cast<int>(len / 8);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.full[b], 1);
            mbar_init(&sm.xfull[b], 1);
        }
        mbar_fence_init();
    }
    __syncthreads();
    // Use k of the slice buffer: expert e's slice, in 16 KiB copies.
    auto load = [&](int e, int k) {
        uint64_t *bar = &sm.full[k & 1];
        mbar_arrive_expect_tx(bar, len);
        const uint8_t *src = scales + static_cast<long long>(e) * per_expert + lo;
        for (uint32_t off = 0; off < len; off += 16384u)
            bulk_load(smem_u32(sm.slice + off), src + off, min(16384u, len - off), bar);
    };
    // Exchange k: block maximum and count, one message to every CTA of the
    // cluster; starts the copy of expert e_next once the slice is free (every
    // thread has passed the block barrier, so it holds its words in registers).
    auto exchange = [&](int k, uint32_t m_warp, uint32_t c_warp, int e_next) {
        if ((tid & 31) == 0) {
            sm.wmax[tid >> 5] = m_warp;
            sm.wcnt[tid >> 5] = c_warp;
        }
        __syncthreads();
        if (tid == 0 && e_next < E) load(e_next, k + 1);
        const int xb = k & 1;
        if (tid < static_cast<int>(C)) {
            uint32_t m = 0, c = 0;
            for (int w = 0; w < kOneNT / 32; ++w) {
                m = max(m, sm.wmax[w]);
                c += sm.wcnt[w];
            }
            if (tid == 0) mbar_arrive_expect_tx(&sm.xfull[xb], 8u * C);
            st_async_v2(cluster_addr(&sm.xch[xb][rank][0], tid), m, c, cluster_addr(&sm.xfull[xb], tid));
        }
        wait_bounded(&sm.xfull[xb], (k >> 1) & 1, nullptr, status, limit_ns);
    };
    auto count_sum = [&](int xb) {
        uint32_t t = 0;
        for (uint32_t r = 0; r < C; ++r) t += sm.xch[xb][r][1];
        return t;
    };
    if (tid == 0 && first < E) load(first, 0);
    // Every CTA's barriers are initialised before a peer's first message.
    cluster_sync();
    uint32_t prev_in_range = 0;            // this thread's count for the previous expert
    int k = 0, e_prev = -1;
    for (int e = first; e < E; e += n_clusters, ++k) {
        if (!wait_bounded(&sm.full[k & 1], (k >> 1) & 1, nullptr, status, limit_ns))
            wait_bounded(&sm.full[k & 1], (k >> 1) & 1, nullptr, nullptr, limit_ns);   // drain
        const uint2 *s = reinterpret_cast<const uint2 *>(sm.slice);
        uint2 v[kOneWords];
        uint32_t acc = 0;
#pragma unroll
        for (int u = 0; u < kOneWords; ++u) {
            const int j = tid + u * kOneNT;
            v[u] = j < nwords ? s[j] : make_uint2(0u, 0u);
            acc = __vmaxu4(acc, __vmaxu4(v[u].x, v[u].y));
        }
        // The next bulk copy (async proxy) overwrites what these reads saw.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        exchange(k, __reduce_max_sync(0xffffffffu, max_byte4(acc)),
                 __reduce_add_sync(0xffffffffu, prev_in_range), e + n_clusters);
        const int xb = k & 1;
        uint32_t m = 0;
        for (uint32_t r = 0; r < C; ++r) m = max(m, sm.xch[xb][r][0]);
        if (rank == 0 && tid == 0) {
            if (e_prev >= 0)
                out_of_range[e_prev] = static_cast<unsigned long long>(per_expert) - count_sum(xb);
            weight_scale_2[e] = weight_scale_2_of(m);
            if (m == 255u) set_status(status, MOE_ERR_DATA);
        }
        const uint32_t M = m * kOnes;
        uint32_t in_range = 0;
        uint4 *dst = reinterpret_cast<uint4 *>(e4m3 + 2 * (static_cast<long long>(e) * per_expert + lo));
        // 8 scale bytes -> 16 output bytes per word: a warp stores 512
        // contiguous bytes per instruction.
#pragma unroll
        for (int u = 0; u < kOneWords; ++u) {
            const int j = tid + u * kOneNT;
            if (j < nwords) {
                const uint32_t a = convert_word(v[u].x, M, in_range);
                const uint32_t b = convert_word(v[u].y, M, in_range);
                __stcs(dst + j, make_uint4(prmt(a, 0u, 0x1100u), prmt(a, 0u, 0x3322u), prmt(b, 0u, 0x1100u),
                                           prmt(b, 0u, 0x3322u)));
            }
        }
        prev_in_range = in_range;
        e_prev = e;
    }
    // The last expert's counts (every cluster has at least one expert).
    if (k > 0) {
        exchange(k, 0u, __reduce_add_sync(0xffffffffu, prev_in_range), E);
        if (rank == 0 && tid == 0)
            out_of_range[e_prev] = static_cast<unsigned long long>(per_expert) - count_sum(k & 1);
    }
    // No CTA leaves while a peer may still address its shared memory.
    cluster_sync();
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
                                 int *kmax_scratch, int *status, uint64_t wait_limit_ns,
                                 cudaStream_t stream, int num_sms, int *launches) {
    using namespace cast;
    *launches = 0;
    const long long per_expert = static_cast<long long>(N) * (K / 32);
    if (nvfp4_cast_one_pass(scales, e4m3, N, K)) {
        const int C = static_cast<int>((per_expert + kSlice - 1) / kSlice);
        const int smem = static_cast<int>(sizeof(OnePassSmem));
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
        // The shared-memory attribute, once per device (0..63; others every call).
        static std::atomic<uint64_t> attr_dev_mask{0};
        const uint64_t dev_bit = dev >= 0 && dev < 64 ? 1ull << dev : 0;
        if (!(attr_dev_mask.load(std::memory_order_acquire) & dev_bit) || !dev_bit) {
            if (cudaFuncSetAttribute(onepass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess)
                return MOE_ERR_CUDA;
            attr_dev_mask.fetch_or(dev_bit, std::memory_order_release);
        }
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(C);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.blockDim = dim3(kOneNT, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cfg.stream = stream;
        // Resident clusters of this size, per device (queried once).
        static std::atomic<int> resident[64][kMaxCluster + 1];
        int nc = dev >= 0 && dev < 64 ? resident[dev][C].load(std::memory_order_relaxed) : 0;
        if (nc <= 0) {
            cfg.gridDim = dim3(static_cast<unsigned>(C * num_sms), 1, 1);
            if (cudaOccupancyMaxActiveClusters(&nc, onepass_kernel, &cfg) != cudaSuccess || nc <= 0)
                return MOE_ERR_CUDA;
            if (dev >= 0 && dev < 64) resident[dev][C].store(nc, std::memory_order_relaxed);
        }
        nc = min(nc, E);
        cfg.gridDim = dim3(static_cast<unsigned>(C * nc), 1, 1);
        if (cudaLaunchKernelEx(&cfg, onepass_kernel, scales, per_expert, E, e4m3, weight_scale_2,
                               out_of_range, status, wait_limit_ns) != cudaSuccess)
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
