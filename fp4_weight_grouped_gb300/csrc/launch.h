// Internal launchers behind the C ABI (host side).  Arguments are already
// validated by api.cu; each launcher only enqueues kernels on `stream`.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_mxfp4.h"

namespace moe {

// Kernel launches per grouped GEMM call: one per band class (bands of up to 32
// rows, and longer bands).
constexpr int kGemmLaunches = 2;

size_t route_sort_scratch_bytes(int T, int k, int E);

moe_status launch_route_sort(const int32_t *ids, int T, int k, int E, int32_t *group_sizes,
                             int32_t *offsets, int32_t *sorted_slot, int32_t *slot_to_row,
                             const uint16_t *x, int hidden, uint16_t *x_sorted, int x_k8,
                             void *scratch, int *status, cudaStream_t stream, int *launches,
                             uint16_t *x_tok = nullptr);

moe_status launch_route_sort_noalloc(const int32_t *ids, int T, int k, int E,
                                     int32_t *group_sizes, int32_t *offsets,
                                     int32_t *sorted_slot, int32_t *slot_to_row,
                                     const uint16_t *x, int hidden, uint16_t *x_sorted, int x_k8,
                                     cudaStream_t stream, int *launches);

moe_status launch_grouped_gemm(const uint16_t *act, int rows, int K, const uint8_t *codes,
                               const uint8_t *scales, const int32_t *group_sizes, int E, int N,
                               void *out, int out_bf16, int act_k8, int *status,
                               uint64_t wait_limit_ns, cudaStream_t stream, int num_sms);

// MXFP4 with one E8M0 scale per scale_block (32 or 512) consecutive k.
moe_status launch_grouped_gemm_block(const uint16_t *act, int rows, int K, int scale_block,
                                     const uint8_t *codes, const uint8_t *scales,
                                     const int32_t *group_sizes, int E, int N, void *out,
                                     int out_bf16, int act_k8, int *status, uint64_t wait_limit_ns,
                                     cudaStream_t stream, int num_sms);

// Fused w13 + SwiGLU: N = 2 * I weight rows ([gate | up]) -> h bf16 [rows, I].
moe_status launch_grouped_gemm_swiglu(const uint16_t *act, int rows, int K, const uint8_t *codes,
                                      const uint8_t *scales, const int32_t *group_sizes, int E,
                                      int N, uint16_t *h, int act_k8, int h_k8, int *status,
                                      uint64_t wait_limit_ns, cudaStream_t stream, int num_sms);

// Fused w13 + SwiGLU with the routing permutation in the activation load:
// sorted row r reads row sorted_slot[r] / top_k of x_k8 [act_rows, K]
// (K8-interleaved token activations).
moe_status launch_grouped_gemm_swiglu_gather(const uint16_t *x_k8, int act_rows, int top_k,
                                             const int32_t *sorted_slot, int rows, int K,
                                             const uint8_t *codes, const uint8_t *scales,
                                             const int32_t *group_sizes, int E, int N, uint16_t *h,
                                             int h_k8, int *status, uint64_t wait_limit_ns,
                                             cudaStream_t stream, int num_sms);

// Grouped GEMM writing sorted row r to output row out_row[r].
moe_status launch_grouped_gemm_scatter(const uint16_t *act, int rows, int K, const uint8_t *codes,
                                       const uint8_t *scales, const int32_t *group_sizes, int E,
                                       int N, const int32_t *out_row, void *out, int out_bf16,
                                       int act_k8, int *status, uint64_t wait_limit_ns,
                                       cudaStream_t stream, int num_sms);

moe_status launch_grouped_gemm_nvfp4(const uint16_t *act, int rows, int K, const uint8_t *codes,
                                     const uint8_t *scales16, const float *weight_scale_2,
                                     const int32_t *group_sizes, int E, int N, void *out,
                                     int out_bf16, int act_k8, int *status,
                                     uint64_t wait_limit_ns, cudaStream_t stream, int num_sms);

// CTA-pair use for bands over 32 rows: 0 automatic, 1 never, 2 whenever the
// shape allows (process-wide).
void set_gemm_pairing(int mode);

moe_status launch_decode_expert(const uint8_t *codes, const uint8_t *scales, int N, int K, int e,
                                uint16_t *out, int *status, cudaStream_t stream);

moe_status launch_mxfp4_to_nvfp4(const uint8_t *scales, int E, int N, int K, uint8_t *e4m3,
                                 float *weight_scale_2, unsigned long long *out_of_range,
                                 int *kmax_scratch, int *status, uint64_t wait_limit_ns,
                                 cudaStream_t stream, int num_sms, int *launches);

moe_status launch_bounded_wait(uint64_t limit_ns, int *status, cudaStream_t stream);

moe_status launch_swiglu(const void *gu, int in_bf16, long long rows, int I, uint16_t *h,
                         int h_k8, cudaStream_t stream, int num_sms);

// x_k8 [rows, hidden] = x with every 8 bf16 in the K8-interleaved order.
moe_status launch_interleave_k8(const uint16_t *x, long long rows, int hidden, uint16_t *x_k8,
                                cudaStream_t stream, int num_sms);

// slot_order: y row of slot s is s (s2r only marks the slots that count).
moe_status launch_combine(const float *y, const int32_t *s2r, const float *w, int T, int k, int N,
                          void *out, int out_bf16, cudaStream_t stream, int num_sms,
                          int slot_order = 0);

}  // namespace moe
