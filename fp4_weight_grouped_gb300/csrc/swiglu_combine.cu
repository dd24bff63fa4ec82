// SwiGLU on the fused w13 output and the deterministic top-k combine.
//
// SwiGLU ("Running DeepSeek V4 Flash on TPU v6", section 1, the gate/up
// activation left out of the grouped-matmul timings; "DeepSeek-V4-Flash-0731-
// NVFP4": w1/w3 fused as GEMM1): h = silu_f32(g) * u with g the first I columns and u
// the next I, in f32, rounded once to bf16.
//
// Combine ("DeepSeek-V4-Flash" (PocketLLM), "Correctness and precision": the MoE
// expert reduction is deterministic, without atomicAdd): out[t] = sum_j
// w[t,j] * y[slot_to_row[t*k+j]] as an f32 FMA chain in ascending j.
//
// With y in slot order (the w2 GEMM's scatter), y row t*k+j is read directly.
//
// K8 interleave of activation rows (the layout the grouped GEMM's decode order
// wants): a permutation inside every 8 bf16.
//
// All are HBM-bound streams: 16-byte vector loads and stores, grid-stride loops
// over a grid sized to a multiple of the SM count.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "launch.h"
#include "mxfp4_decode.cuh"

namespace moe {
namespace ew {

__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

template <typename T>
__global__ void swiglu_vec8(const T *gu, long long rows, int I, uint16_t *h, int h_k8) {
    const int per_row = I / 8;
    const long long total = rows * per_row;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = idx / per_row;
        const int i = static_cast<int>(idx - r * per_row) * 8;
        const T *row = gu + r * 2 * static_cast<long long>(I);
        float g[8], u[8];
        load8(row + i, g);
        load8(row + I + i, u);
        uint4 o;
        o.x = pack_bf16x2(silu_f32(g[0]) * u[0], silu_f32(g[1]) * u[1]);
        o.y = pack_bf16x2(silu_f32(g[2]) * u[2], silu_f32(g[3]) * u[3]);
        o.z = pack_bf16x2(silu_f32(g[4]) * u[4], silu_f32(g[5]) * u[5]);
        o.w = pack_bf16x2(silu_f32(g[6]) * u[6], silu_f32(g[7]) * u[7]);
        *reinterpret_cast<uint4 *>(h + r * I + i) = h_k8 ? interleave8(o) : o;
    }
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__global__ void swiglu_scalar(const T *gu, long long rows, int I, uint16_t *h) {
    const long long total = rows * I;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = idx / I;
        const int i = static_cast<int>(idx - r * I);
        const float g = to_f32(gu[r * 2 * I + i]);
        const float u = to_f32(gu[r * 2 * I + I + i]);
        const __nv_bfloat16 b = __float2bfloat16_rn(silu_f32(g) * u);
        h[idx] = *reinterpret_cast<const uint16_t *>(&b);
    }
}

// One token row per block iteration; each thread owns 4 consecutive columns.
// y rows in sorted order (row s2r[slot]) or, with slot_order, in slot order
// (row = slot); either way a slot with s2r outside [0, T*k) adds nothing.
template <bool OUT_BF16>
__global__ void combine_vec4(const float *y, const int32_t *s2r, const float *w, int T, int k,
                             int N, void *out, int slot_order) {
    const int n4 = N / 4;
    const int rows = T * k;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        for (int c = threadIdx.x; c < n4; c += blockDim.x) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < k; ++j) {
                const int slot = t * k + j;
                const int r = __ldg(s2r + slot);
                // A slot whose id was out of range has no row (-1): it adds nothing.
                if (static_cast<unsigned>(r) >= static_cast<unsigned>(rows)) continue;
                const int row = slot_order ? slot : r;
                const float wj = __ldg(w + static_cast<size_t>(t) * k + j);
                const float4 v = __ldg(reinterpret_cast<const float4 *>(y + static_cast<size_t>(row) * N) + c);
                acc.x = fmaf(wj, v.x, acc.x);
                acc.y = fmaf(wj, v.y, acc.y);
                acc.z = fmaf(wj, v.z, acc.z);
                acc.w = fmaf(wj, v.w, acc.w);
            }
            if (OUT_BF16) {
                uint2 o;
                o.x = pack_bf16x2(acc.x, acc.y);
                o.y = pack_bf16x2(acc.z, acc.w);
                reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + static_cast<size_t>(t) * N)[c] = o;
            } else {
                reinterpret_cast<float4 *>(static_cast<float *>(out) + static_cast<size_t>(t) * N)[c] = acc;
            }
        }
    }
}

template <bool OUT_BF16>
__global__ void combine_scalar(const float *y, const int32_t *s2r, const float *w, int T, int k,
                               int N, void *out, int slot_order) {
    const int rows = T * k;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        for (int n = threadIdx.x; n < N; n += blockDim.x) {
            float acc = 0.f;
            for (int j = 0; j < k; ++j) {
                const int slot = t * k + j;
                const int r = s2r[slot];
                if (static_cast<unsigned>(r) >= static_cast<unsigned>(rows)) continue;
                const int row = slot_order ? slot : r;
                acc = fmaf(w[static_cast<size_t>(t) * k + j], y[static_cast<size_t>(row) * N + n], acc);
            }
            if (OUT_BF16) {
                const __nv_bfloat16 b = __float2bfloat16_rn(acc);
                static_cast<uint16_t *>(out)[static_cast<size_t>(t) * N + n] =
                    *reinterpret_cast<const uint16_t *>(&b);
            } else {
                static_cast<float *>(out)[static_cast<size_t>(t) * N + n] = acc;
            }
        }
    }
}

__global__ void interleave_k8_vec8(const uint4 *x, long long n16, uint4 *out) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        out[i] = interleave8(__ldg(x + i));
}

}  // namespace ew

moe_status launch_interleave_k8(const uint16_t *x, long long rows, int hidden, uint16_t *x_k8,
                                cudaStream_t stream, int num_sms) {
    const long long n16 = rows * (hidden / 8);
    if (n16 == 0) return MOE_OK;
    long long blocks = (n16 + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    ew::interleave_k8_vec8<<<static_cast<int>(blocks), 256, 0, stream>>>(
        reinterpret_cast<const uint4 *>(x), n16, reinterpret_cast<uint4 *>(x_k8));
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_swiglu(const void *gu, int in_bf16, long long rows, int I, uint16_t *h,
                         int h_k8, cudaStream_t stream, int num_sms) {
    if (rows == 0 || I == 0) return MOE_OK;
    const bool vec = (I % 8) == 0;
    const long long work = vec ? rows * (I / 8) : rows * I;
    long long blocks = (work + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (vec) {
        if (in_bf16)
            ew::swiglu_vec8<<<static_cast<int>(blocks), 256, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(gu), rows, I, h, h_k8);
        else
            ew::swiglu_vec8<<<static_cast<int>(blocks), 256, 0, stream>>>(
                static_cast<const float *>(gu), rows, I, h, h_k8);
    } else {
        if (in_bf16)
            ew::swiglu_scalar<<<static_cast<int>(blocks), 256, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(gu), rows, I, h);
        else
            ew::swiglu_scalar<<<static_cast<int>(blocks), 256, 0, stream>>>(
                static_cast<const float *>(gu), rows, I, h);
    }
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_combine(const float *y, const int32_t *s2r, const float *w, int T, int k, int N,
                          void *out, int out_bf16, cudaStream_t stream, int num_sms,
                          int slot_order) {
    if (T == 0 || N == 0) return MOE_OK;
    int blocks = T < num_sms * 16 ? T : num_sms * 16;
    const bool vec = (N % 4) == 0;
    const int threads = vec ? (N / 4 < 256 ? ((N / 4 + 31) / 32) * 32 : 256) : 256;
    if (vec) {
        if (out_bf16) ew::combine_vec4<true><<<blocks, threads, 0, stream>>>(y, s2r, w, T, k, N, out, slot_order);
        else ew::combine_vec4<false><<<blocks, threads, 0, stream>>>(y, s2r, w, T, k, N, out, slot_order);
    } else {
        if (out_bf16) ew::combine_scalar<true><<<blocks, threads, 0, stream>>>(y, s2r, w, T, k, N, out, slot_order);
        else ew::combine_scalar<false><<<blocks, threads, 0, stream>>>(y, s2r, w, T, k, N, out, slot_order);
    }
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
