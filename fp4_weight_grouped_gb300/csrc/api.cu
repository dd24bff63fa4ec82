// C ABI of the library: argument validation, device checks and launches.
// See include/moe_mxfp4.h for the contract of every entry point.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/moe_mxfp4.h"
#include "launch.h"

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per pipeline wait
constexpr int kMaxE = 1024;
constexpr size_t kStatusBytes = 256;

thread_local int32_t g_last_launches = 0;

// Per device: 0 not yet looked up, -1 not compute capability 10.3, else its
// SM count.  Host threads may race on the first lookup; each stores the same
// value, published with release and read with acquire.
std::atomic<int> g_dev_sms[64];

// Current device must be compute capability 10.3 (GB300).
moe_status current_device(int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    int sms = g_dev_sms[dev].load(std::memory_order_acquire);
    if (sms == 0) {
        int major = 0, minor = 0, count = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        sms = (major == 10 && minor == 3 && count > 0) ? count : -1;
        g_dev_sms[dev].store(sms, std::memory_order_release);
    }
    if (sms < 0) return MOE_ERR_UNSUPPORTED;
    *num_sms = sms;
    return MOE_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int *status_word(void *workspace) { return static_cast<int *>(workspace); }

moe_status check_gemm_args(const uint16_t *act, int layout, int64_t rows, int32_t K, const uint8_t *codes,
                           const uint8_t *scales, const int32_t *group_sizes, int32_t E, int32_t N,
                           const void *out, moe_dtype out_dtype, const void *workspace,
                           size_t workspace_bytes) {
    if (rows < 0 || rows > INT32_MAX || K <= 0 || K % 32 != 0 || N <= 0 || E <= 0 || E > kMaxE)
        return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(E) * N > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_F32 && out_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (layout != MOE_ACT_ROW_MAJOR && layout != MOE_ACT_K8_INTERLEAVED) return MOE_ERR_INVALID_ARG;
    if (!codes || !scales || !group_sizes || !workspace || workspace_bytes < kStatusBytes)
        return MOE_ERR_INVALID_ARG;
    if (rows > 0 && (!act || !out)) return MOE_ERR_INVALID_ARG;
    if (!aligned(act, 16) || !aligned(codes, 16) || !aligned(workspace, 16))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(out, out_dtype == MOE_F32 ? 4 : 2)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status check_route_args(const int32_t *ids, int32_t T, int32_t k, int32_t E,
                            const int32_t *gs, const int32_t *off, const int32_t *ss,
                            const int32_t *s2r, const uint16_t *x, int32_t hidden,
                            const uint16_t *xs, int layout, const void *workspace,
                            size_t workspace_bytes) {
    if (T < 0 || E <= 0 || E > kMaxE || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * k > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (!gs || !off || !workspace) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!ids || !ss || !s2r)) return MOE_ERR_INVALID_ARG;
    if ((x == nullptr) != (xs == nullptr)) return MOE_ERR_INVALID_ARG;
    if (layout != MOE_ACT_ROW_MAJOR && layout != MOE_ACT_K8_INTERLEAVED &&
        layout != MOE_ACT_K8_TOKEN_ORDER)
        return MOE_ERR_INVALID_ARG;
    if (x && (hidden <= 0 || hidden % 8 != 0 || !aligned(x, 16) || !aligned(xs, 16)))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(workspace, 16) || workspace_bytes < moe_workspace_bytes(T, k, E))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

extern "C" {

const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DATA: return "MOE_ERR_DATA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
    }
    return "MOE_ERR_UNKNOWN";
}

size_t moe_workspace_bytes(int32_t T, int32_t k, int32_t E) {
    if (T < 0 || k < 0 || E < 0) return kStatusBytes;
    return kStatusBytes + moe::route_sort_scratch_bytes(T, k, E);
}

moe_status moe_clear_status(void *workspace, void *stream) {
    if (!workspace) return MOE_ERR_INVALID_ARG;
    g_last_launches = 0;
    return cudaMemsetAsync(workspace, 0, sizeof(int), static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

moe_status moe_read_status(const void *workspace, void *stream) {
    if (!workspace) return MOE_ERR_INVALID_ARG;
    int v = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return static_cast<moe_status>(v);
}

moe_status moe_route_sort(const int32_t *topk_ids, int32_t T, int32_t k, int32_t E,
                          int32_t *group_sizes, int32_t *group_offsets, int32_t *sorted_slot,
                          int32_t *slot_to_row, const uint16_t *x, int32_t hidden,
                          uint16_t *x_sorted, moe_act_layout x_sorted_layout, void *workspace,
                          size_t workspace_bytes, void *stream) {
    moe_status st = check_route_args(topk_ids, T, k, E, group_sizes, group_offsets, sorted_slot,
                                     slot_to_row, x, hidden, x_sorted, x_sorted_layout, workspace,
                                     workspace_bytes);
    if (st != MOE_OK) return st;
    int sms = 0;
    if ((st = current_device(&sms)) != MOE_OK) return st;
    int launches = 0;
    const bool tokens = x_sorted_layout == MOE_ACT_K8_TOKEN_ORDER;
    st = moe::launch_route_sort(topk_ids, T, k, E, group_sizes, group_offsets, sorted_slot,
                                slot_to_row, x, hidden, tokens ? nullptr : x_sorted,
                                x_sorted_layout == MOE_ACT_K8_INTERLEAVED,
                                static_cast<uint8_t *>(workspace) + kStatusBytes,
                                status_word(workspace), static_cast<cudaStream_t>(stream),
                                &launches, tokens ? x_sorted : nullptr);
    g_last_launches = launches;
    return st;
}

moe_status moe_route_sort_noalloc(const int32_t *topk_ids, int32_t T, int32_t k, int32_t E,
                                  int32_t *group_sizes, int32_t *group_offsets,
                                  int32_t *sorted_slot, int32_t *slot_to_row, const uint16_t *x,
                                  int32_t hidden, uint16_t *x_sorted,
                                  moe_act_layout x_sorted_layout, void *stream) {
    // The checks of moe_route_sort that do not concern the workspace.
    if (T < 0 || E <= 0 || E > kMaxE || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * k > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (!group_sizes || !group_offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !sorted_slot || !slot_to_row)) return MOE_ERR_INVALID_ARG;
    if ((x == nullptr) != (x_sorted == nullptr)) return MOE_ERR_INVALID_ARG;
    if (x_sorted_layout != MOE_ACT_ROW_MAJOR && x_sorted_layout != MOE_ACT_K8_INTERLEAVED)
        return MOE_ERR_INVALID_ARG;
    if (x && (hidden <= 0 || hidden % 8 != 0 || !aligned(x, 16) || !aligned(x_sorted, 16)))
        return MOE_ERR_INVALID_ARG;
    if (moe::route_sort_scratch_bytes(T, k, E) > MOE_ROUTE_SORT_NOALLOC_SCRATCH_BYTES)
        return MOE_ERR_CAPACITY;
    int sms = 0;
    moe_status st = current_device(&sms);
    if (st != MOE_OK) return st;
    int launches = 0;
    st = moe::launch_route_sort_noalloc(topk_ids, T, k, E, group_sizes, group_offsets,
                                        sorted_slot, slot_to_row, x, hidden, x_sorted,
                                        x_sorted_layout == MOE_ACT_K8_INTERLEAVED,
                                        static_cast<cudaStream_t>(stream), &launches);
    g_last_launches = launches;
    return st;
}

moe_status moe_mxfp4_grouped_gemm(const uint16_t *act, moe_act_layout act_layout, int64_t rows,
                                  int32_t K, const uint8_t *codes, const uint8_t *scales,
                                  const int32_t *group_sizes, int32_t E, int32_t N, void *out,
                                  moe_dtype out_dtype, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    moe_status st = check_gemm_args(act, act_layout, rows, K, codes, scales, group_sizes, E, N,
                                    out, out_dtype, workspace, workspace_bytes);
    if (st != MOE_OK) return st;
    int sms = 0;
    if ((st = current_device(&sms)) != MOE_OK) return st;
    st = moe::launch_grouped_gemm(act, static_cast<int>(rows), K, codes, scales, group_sizes, E, N,
                                  out, out_dtype == MOE_BF16, act_layout == MOE_ACT_K8_INTERLEAVED,
                                  status_word(workspace), kWaitLimitNs,
                                  static_cast<cudaStream_t>(stream), sms);
    g_last_launches = rows > 0 ? moe::kGemmLaunches : 0;
    return st;
}

moe_status moe_mxfp4_grouped_gemm_block(const uint16_t *act, moe_act_layout act_layout,
                                        int64_t rows, int32_t K, int32_t scale_block,
                                        const uint8_t *codes, const uint8_t *scales,
                                        const int32_t *group_sizes, int32_t E, int32_t N,
                                        void *out, moe_dtype out_dtype, void *workspace,
                                        size_t workspace_bytes, void *stream) {
    if ((scale_block != 32 && scale_block != 512) || K <= 0 || K % scale_block != 0)
        return MOE_ERR_INVALID_ARG;
    moe_status st = check_gemm_args(act, act_layout, rows, K, codes, scales, group_sizes, E, N,
                                    out, out_dtype, workspace, workspace_bytes);
    if (st != MOE_OK) return st;
    int sms = 0;
    if ((st = current_device(&sms)) != MOE_OK) return st;
    st = moe::launch_grouped_gemm_block(act, static_cast<int>(rows), K, scale_block, codes, scales,
                                        group_sizes, E, N, out, out_dtype == MOE_BF16,
                                        act_layout == MOE_ACT_K8_INTERLEAVED,
                                        status_word(workspace), kWaitLimitNs,
                                        static_cast<cudaStream_t>(stream), sms);
    g_last_launches = rows > 0 ? moe::kGemmLaunches : 0;
    return st;
}

moe_status moe_mxfp4_grouped_gemm_swiglu(const uint16_t *act, moe_act_layout act_layout,
                                         int64_t rows, int32_t K, const uint8_t *codes,
                                         const uint8_t *scales, const int32_t *group_sizes,
                                         int32_t E, int32_t I, uint16_t *h,
                                         moe_act_layout h_layout, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    if (I <= 0 || I % 16 != 0 || static_cast<int64_t>(I) * 2 > INT32_MAX) return MOE_ERR_INVALID_ARG;
    moe_status st = check_gemm_args(act, act_layout, rows, K, codes, scales, group_sizes, E, 2 * I,
                                    h, MOE_BF16, workspace, workspace_bytes);
    if (st != MOE_OK) return st;
    if (h_layout != MOE_ACT_ROW_MAJOR && (h_layout != MOE_ACT_K8_INTERLEAVED || I % 8 != 0))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = current_device(&sms)) != MOE_OK) return st;
    st = moe::launch_grouped_gemm_swiglu(act, static_cast<int>(rows), K, codes, scales, group_sizes,
                                         E, 2 * I, h, act_layout == MOE_ACT_K8_INTERLEAVED,
                                         h_layout == MOE_ACT_K8_INTERLEAVED,
                                         status_word(workspace), kWaitLimitNs,
                                         static_cast<cudaStream_t>(stream), sms);
    g_last_launches = rows > 0 ? moe::kGemmLaunches : 0;
    return st;
}

moe_status moe_mxfp4_grouped_gemm_swiglu_gather(const uint16_t *x_k8, int32_t T, int32_t top_k,
                                                const int32_t *sorted_slot, int64_t rows, int32_t K,
                                                const uint8_t *codes, const uint8_t *scales,
                                                const int32_t *group_sizes, int32_t E, int32_t I,
                                                uint16_t *h, moe_act_layout h_layout,
                                                void *workspace, size_t workspace_bytes,
                                                void *stream) {
    if (I <= 0 || I % 16 != 0 || static_cast<int64_t>(I) * 2 > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (T < 0 || top_k <= 0 || (rows > 0 && (T == 0 || !sorted_slot))) return MOE_ERR_INVALID_ARG;
    moe_status st = check_gemm_args(x_k8, MOE_ACT_K8_INTERLEAVED, rows, K, codes, scales,
                                    group_sizes, E, 2 * I, h, MOE_BF16, workspace, workspace_bytes);
    if (st != MOE_OK) return st;
    if (h_layout != MOE_ACT_ROW_MAJOR && (h_layout != MOE_ACT_K8_INTERLEAVED || I % 8 != 0))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = current_device(&sms)) != MOE_OK) return st;
    st = moe::launch_grouped_gemm_swiglu_gather(x_k8, T, top_k, sorted_slot, static_cast<int>(rows), K,
                                                codes, scales, group_sizes, E, 2 * I, h,
                                                h_layout == MOE_ACT_K8_INTERLEAVED,
                                                status_word(workspace), kWaitLimitNs,
                                                static_cast<cudaStream_t>(stream), sms);
    g_last_launches = rows > 0 ? moe::kGemmLaunches : 0;
    return st;
}

moe_status moe_mxfp4_grouped_gemm_scatter(const uint16_t *act, moe_act_layout act_layout,
                                          int64_t rows, int32_t K, const uint8_t *codes,
                                          const uint8_t *scales, const int32_t *group_sizes,
                                          int32_t E, int32_t N, const int32_t *out_row, void *out,
                                          moe_dtype out_dtype, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    moe_status st = check_gemm_args(act, act_layout, rows, K, codes, scales, group_sizes, E, N,
                                    out, out_dtype, workspace, workspace_bytes);
    if (st != MOE_OK) return st;
    if (rows > 0 && !out_row) return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = current_device(&sms)) != MOE_OK) return st;
    st = moe::launch_grouped_gemm_scatter(act, static_cast<int>(rows), K, codes, scales, group_sizes,
                                          E, N, out_row, out, out_dtype == MOE_BF16,
                                          act_layout == MOE_ACT_K8_INTERLEAVED,
                                          status_word(workspace), kWaitLimitNs,
                                          static_cast<cudaStream_t>(stream), sms);
    g_last_launches = rows > 0 ? moe::kGemmLaunches : 0;
    return st;
}

moe_status moe_nvfp4_grouped_gemm(const uint16_t *act, moe_act_layout act_layout, int64_t rows,
                                  int32_t K, const uint8_t *codes, const uint8_t *scales16,
                                  const float *weight_scale_2, const int32_t *group_sizes,
                                  int32_t E, int32_t N, void *out, moe_dtype out_dtype,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    moe_status st = check_gemm_args(act, act_layout, rows, K, codes, scales16, group_sizes, E, N,
                                    out, out_dtype, workspace, workspace_bytes);
    if (st != MOE_OK) return st;
    if (!weight_scale_2 || !aligned(weight_scale_2, 4)) return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = current_device(&sms)) != MOE_OK) return st;
    st = moe::launch_grouped_gemm_nvfp4(act, static_cast<int>(rows), K, codes, scales16,
                                        weight_scale_2, group_sizes, E, N, out,
                                        out_dtype == MOE_BF16,
                                        act_layout == MOE_ACT_K8_INTERLEAVED,
                                        status_word(workspace), kWaitLimitNs,
                                        static_cast<cudaStream_t>(stream), sms);
    g_last_launches = rows > 0 ? moe::kGemmLaunches : 0;
    return st;
}

moe_status moe_swiglu(const void *gu, moe_dtype in_dtype, int64_t rows, int32_t I, uint16_t *h,
                      moe_act_layout h_layout, void *stream) {
    if (rows < 0 || I <= 0 || (in_dtype != MOE_F32 && in_dtype != MOE_BF16))
        return MOE_ERR_INVALID_ARG;
    if (h_layout != MOE_ACT_ROW_MAJOR && (h_layout != MOE_ACT_K8_INTERLEAVED || I % 8 != 0))
        return MOE_ERR_INVALID_ARG;
    if (rows > 0 && (!gu || !h || !aligned(gu, 16) || !aligned(h, 16))) return MOE_ERR_INVALID_ARG;
    int sms = 0;
    moe_status st = current_device(&sms);
    if (st != MOE_OK) return st;
    st = moe::launch_swiglu(gu, in_dtype == MOE_BF16, rows, I, h,
                            h_layout == MOE_ACT_K8_INTERLEAVED, static_cast<cudaStream_t>(stream),
                            sms);
    g_last_launches = rows > 0 ? 1 : 0;
    return st;
}

moe_status moe_combine(const float *y, const int32_t *slot_to_row, const float *topk_w,
                       int32_t T, int32_t k, int32_t N, void *out, moe_dtype out_dtype,
                       void *stream) {
    if (T < 0 || k <= 0 || N <= 0 || (out_dtype != MOE_F32 && out_dtype != MOE_BF16))
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!y || !slot_to_row || !topk_w || !out || !aligned(y, 16) || !aligned(out, 16)))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    moe_status st = current_device(&sms);
    if (st != MOE_OK) return st;
    st = moe::launch_combine(y, slot_to_row, topk_w, T, k, N, out, out_dtype == MOE_BF16,
                             static_cast<cudaStream_t>(stream), sms);
    g_last_launches = T > 0 ? 1 : 0;
    return st;
}

moe_status moe_combine_slots(const float *y, const int32_t *slot_to_row, const float *topk_w,
                             int32_t T, int32_t k, int32_t N, void *out, moe_dtype out_dtype,
                             void *stream) {
    if (T < 0 || k <= 0 || N <= 0 || (out_dtype != MOE_F32 && out_dtype != MOE_BF16))
        return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * k > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!y || !slot_to_row || !topk_w || !out || !aligned(y, 16) || !aligned(out, 16)))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    moe_status st = current_device(&sms);
    if (st != MOE_OK) return st;
    st = moe::launch_combine(y, slot_to_row, topk_w, T, k, N, out, out_dtype == MOE_BF16,
                             static_cast<cudaStream_t>(stream), sms, 1);
    g_last_launches = T > 0 ? 1 : 0;
    return st;
}

moe_status moe_act_interleave_k8(const uint16_t *x, int64_t rows, int32_t hidden, uint16_t *x_k8,
                                 void *stream) {
    if (rows < 0 || hidden <= 0 || hidden % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (rows > 0 && (!x || !x_k8 || !aligned(x, 16) || !aligned(x_k8, 16)))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    moe_status st = current_device(&sms);
    if (st != MOE_OK) return st;
    st = moe::launch_interleave_k8(x, rows, hidden, x_k8, static_cast<cudaStream_t>(stream), sms);
    g_last_launches = rows > 0 ? 1 : 0;
    return st;
}

moe_status moe_layer_forward(const uint16_t *x, const int32_t *topk_ids, const float *topk_w,
                             int32_t T, int32_t k, int32_t E, int32_t hidden, int32_t inter,
                             const uint8_t *w13_codes, const uint8_t *w13_scales,
                             const uint8_t *w2_codes, const uint8_t *w2_scales, float *out,
                             int32_t *group_sizes, int32_t *group_offsets, int32_t *sorted_slot,
                             int32_t *slot_to_row, uint16_t *x_sorted, uint16_t *h, float *y2,
                             void *workspace, size_t workspace_bytes, void *stream) {
    if (hidden <= 0 || inter <= 0 || hidden % 32 || inter % 32) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(inter) * 2 > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !out || !x_sorted || !h || !y2 || !topk_w)) return MOE_ERR_INVALID_ARG;
    const int64_t rows = static_cast<int64_t>(T) * k;
    moe_status st = check_route_args(topk_ids, T, k, E, group_sizes, group_offsets, sorted_slot,
                                     slot_to_row, x, hidden, x_sorted, MOE_ACT_K8_INTERLEAVED,
                                     workspace, workspace_bytes);
    if (st != MOE_OK) return st;
    if ((st = check_gemm_args(x_sorted, MOE_ACT_K8_INTERLEAVED, rows, hidden, w13_codes,
                              w13_scales, group_sizes, E, 2 * inter, h, MOE_BF16, workspace,
                              workspace_bytes)) != MOE_OK ||
        (st = check_gemm_args(h, MOE_ACT_K8_INTERLEAVED, rows, inter, w2_codes, w2_scales,
                              group_sizes, E, hidden, y2, MOE_F32, workspace, workspace_bytes)) !=
            MOE_OK)
        return st;
    if (T > 0 && (!aligned(h, 16) || !aligned(y2, 16) || !aligned(out, 16)))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = current_device(&sms)) != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0, n = 0;
    int *status = status_word(workspace);
    st = moe::launch_route_sort(topk_ids, T, k, E, group_sizes, group_offsets, sorted_slot,
                                slot_to_row, x, hidden, x_sorted, 1,
                                static_cast<uint8_t *>(workspace) + kStatusBytes, status, s, &n);
    launches += n;
    if (st == MOE_OK && rows > 0) {   // w13 with SwiGLU in its epilogue: h, never y13
        st = moe::launch_grouped_gemm_swiglu(x_sorted, static_cast<int>(rows), hidden, w13_codes,
                                             w13_scales, group_sizes, E, 2 * inter, h, 1, 1,
                                             status, kWaitLimitNs, s, sms);
        launches += moe::kGemmLaunches;
    }
    if (st == MOE_OK && rows > 0) {
        st = moe::launch_grouped_gemm(h, static_cast<int>(rows), inter, w2_codes, w2_scales,
                                      group_sizes, E, hidden, y2, 0, 1, status, kWaitLimitNs, s,
                                      sms);
        launches += moe::kGemmLaunches;
    }
    if (st == MOE_OK && T > 0) {
        st = moe::launch_combine(y2, slot_to_row, topk_w, T, k, hidden, out, 0, s, sms);
        ++launches;
    }
    g_last_launches = launches;
    return st;
}

moe_status moe_set_gemm_pairing(int32_t mode) {
    if (mode < MOE_PAIRING_AUTO || mode > MOE_PAIRING_ON) return MOE_ERR_INVALID_ARG;
    moe::set_gemm_pairing(mode);
    return MOE_OK;
}

moe_status moe_mxfp4_decode_expert(const uint8_t *codes, const uint8_t *scales, int32_t E,
                                   int32_t N, int32_t K, int32_t e, uint16_t *out,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    if (!codes || !scales || !out || !workspace || workspace_bytes < kStatusBytes || E <= 0 ||
        N <= 0 || K <= 0 || K % 32 || e < 0 || e >= E || !aligned(out, 4))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    moe_status st = current_device(&sms);
    if (st != MOE_OK) return st;
    st = moe::launch_decode_expert(codes, scales, N, K, e, out, status_word(workspace),
                                   static_cast<cudaStream_t>(stream));
    g_last_launches = 1;
    return st;
}

size_t moe_nvfp4_cast_workspace_bytes(int32_t E) {
    return E <= 0 ? kStatusBytes : kStatusBytes + ((static_cast<size_t>(E) * sizeof(int) + 255) & ~size_t(255));
}

moe_status moe_mxfp4_to_nvfp4(const uint8_t *scales, int32_t E, int32_t N, int32_t K,
                              uint8_t *e4m3_scales, float *weight_scale_2, uint64_t *out_of_range,
                              void *workspace, size_t workspace_bytes, void *stream) {
    if (!scales || !e4m3_scales || !weight_scale_2 || !out_of_range || !workspace || E <= 0 ||
        E > 65535 || N <= 0 || K <= 0 || K % 32 || !aligned(workspace, 16) ||
        !aligned(weight_scale_2, 4) || !aligned(out_of_range, 8) ||
        workspace_bytes < moe_nvfp4_cast_workspace_bytes(E))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    moe_status st = current_device(&sms);
    if (st != MOE_OK) return st;
    int launches = 0;
    st = moe::launch_mxfp4_to_nvfp4(
        scales, E, N, K, e4m3_scales, weight_scale_2,
        reinterpret_cast<unsigned long long *>(out_of_range),
        reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) + kStatusBytes),
        status_word(workspace), kWaitLimitNs, static_cast<cudaStream_t>(stream), sms, &launches);
    g_last_launches = launches;
    return st;
}

moe_status moe_debug_bounded_wait(uint64_t limit_ns, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (!workspace || workspace_bytes < kStatusBytes || limit_ns < 1000 ||
        limit_ns > 5000000000ull)
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    moe_status st = current_device(&sms);
    if (st != MOE_OK) return st;
    st = moe::launch_bounded_wait(limit_ns, status_word(workspace),
                                  static_cast<cudaStream_t>(stream));
    g_last_launches = 1;
    return st;
}

int32_t moe_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
