/*
 * moe_mxfp4.h — C ABI of the GB300 (sm_103a) MXFP4 grouped MoE library.
 *
 * The library runs the routed-expert hot path of a DeepSeek-V4-Flash-style MoE
 * layer: tokens routed top-k, sorted into one contiguous row band per expert,
 * multiplied by that expert's MXFP4 weights (W4A16), gated by SwiGLU, multiplied
 * again, and reduced back per token.  The operations follow:
 *
 *  [TPU]    "Running DeepSeek V4 Flash on TPU v6", section 1 "Four bits that v6e
 *           can't hold": expert-sorted row bands, the grouped-matmul loop nest
 *           (N tiles, (expert, M tile) pairs, K inner, f32 accumulator), the e2m1
 *           decode (magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6), per-32 block scales
 *           applied before the matmul, bf16 activations, ragged groups with
 *           empty ones, gate/up (w13) and w2 shapes.
 *  [NVFP4]  "DeepSeek-V4-Flash-0731-NVFP4", "The lossless weight cast": E8M0
 *           per-32 power-of-two scales, fused w1/w3, E2M1 -0 read as +0.
 *  [Pocket] "DeepSeek-V4-Flash" (PocketLLM), "Implemented execution paths" and
 *           "Correctness and precision": deterministic expert reduction with no
 *           atomicAdd.
 *
 * Conventions for every call:
 *  - Pointers named as device buffers must be device memory of the current
 *    CUDA device; the caller owns all of them.  The library allocates nothing
 *    and keeps no state between calls, apart from the fixed scratch array of
 *    moe_route_sort_noalloc.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call only enqueues work on it and returns; results are ready when
 *    the stream reaches that point.
 *  - bf16 values travel as their raw 16-bit patterns (uint16_t); nothing is
 *    converted on the host.
 *  - Return value: argument errors found on the host (null pointer, bad size,
 *    misalignment, unsupported device) and launch failures are returned
 *    synchronously.  Errors that depend on device data (an expert id out of
 *    range, group sizes that do not add up, a scale byte the format does not
 *    allow, a pipeline wait that gave up) are recorded in the status word of
 *    the caller's workspace and read with moe_read_status().  The first error
 *    recorded wins.
 *  - Only compute capability 10.3 (GB300, sm_103a) is supported.
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or dtype (host check) */
    MOE_ERR_UNSUPPORTED = 2, /* device is not compute capability 10.3 */
    MOE_ERR_CUDA = 3,        /* a CUDA runtime/driver call or launch failed */
    MOE_ERR_DATA = 4,        /* device-side: id out of range, sum(group_sizes) != rows,
                                negative group size, an E8M0 scale byte > 252 in the
                                MXFP4 GEMM or 255 in the cast, or an E4M3 NaN scale
                                in the NVFP4 GEMM */
    MOE_ERR_TIMEOUT = 5,     /* device-side: a pipeline wait exceeded its bound */
    MOE_ERR_CAPACITY = 6     /* host check: the problem needs more scratch than a
                                fixed-capacity entry point holds */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Order of the reduction dimension of a bf16 activation matrix [rows, K].
 *  MOE_ACT_ROW_MAJOR      element k of a row at position k.
 *  MOE_ACT_K8_INTERLEAVED within every group of 8 consecutive k (8g .. 8g+7)
 *                         the stored order is 8g + {0,4,1,5,2,6,3,7}; K % 8 == 0.
 *  MOE_ACT_K8_TOKEN_ORDER (moe_route_sort's x output only) x itself, in token
 *                         order [T, hidden], K8-interleaved, instead of the
 *                         gathered copy: the input of
 *                         moe_mxfp4_grouped_gemm_swiglu_gather.
 * The grouped GEMM reduces in the interleaved order (its weight decode pairs
 * codes j and j+4 of every 8); route sort and SwiGLU can write it at no cost,
 * and the GEMM interleaves row-major input itself in shared memory. */
typedef enum {
    MOE_ACT_ROW_MAJOR = 0,
    MOE_ACT_K8_INTERLEAVED = 1,
    MOE_ACT_K8_TOKEN_ORDER = 2
} moe_act_layout;

/* Human-readable name of a status code (static string). */
MOE_API const char *moe_status_string(moe_status status);

/* Bytes of device workspace needed by moe_route_sort for T tokens, top-k and E
 * experts; at least 256 (the status word lives in the first 4 bytes).  The GEMM
 * and the combine only use the status word, so any workspace >= 256 bytes
 * serves them. */
MOE_API size_t moe_workspace_bytes(int32_t T, int32_t k, int32_t E);

/* Clear the status word (async memset of the first 4 bytes of `workspace`).
 * A fresh workspace must be cleared once before first use. */
MOE_API moe_status moe_clear_status(void *workspace, void *stream);

/* Synchronise `stream`, then return the status word recorded in `workspace`
 * (MOE_OK if no device-side error was recorded).  Does not clear it. */
MOE_API moe_status moe_read_status(const void *workspace, void *stream);

/*
 * moe_route_sort — expert-sorted row order for top-k routing ([TPU] section 1:
 * the token rows are ordered by expert so that each expert owns one contiguous
 * band of activation rows), by a stable counting sort.
 *
 *  topk_ids     device int32 [T, k]: expert of routing slot s = t*k + j.
 *  T, k, E      tokens (>= 0), choices per token (1..E), experts (1..1024).
 *  group_sizes  device int32 [E] out: rows per expert (0 allowed).
 *  group_offsets device int32 [E+1] out: exclusive prefix sum; last = T*k.
 *  sorted_slot  device int32 [T*k] out: row -> slot.  Within an expert the
 *               slots appear in ascending s (stable).
 *  slot_to_row  device int32 [T*k] out: slot -> row (inverse of sorted_slot).
 *  x            device bf16 [T, hidden] or NULL: token activations.
 *  hidden       row length of x (multiple of 8 when x is given).
 *  x_sorted     device bf16 [T*k, hidden] out, or NULL: x_sorted[row] =
 *               x[sorted_slot[row] / k] (the activation permutation), x row-major.
 *               With MOE_ACT_K8_TOKEN_ORDER: [T, hidden], x_sorted[t] = x[t] in
 *               the K8 order (no permutation; the gather GEMM does it).
 *  x_sorted_layout  order of the reduction dimension written to x_sorted.
 *  workspace    device, >= moe_workspace_bytes(T, k, E) bytes, 16-byte aligned.
 * Ids outside [0, E) set MOE_ERR_DATA.  Such a slot is left out of every
 * band: slot_to_row holds -1 for it, group_offsets[E] < T*k, and the rows
 * past group_offsets[E] of sorted_slot and x_sorted are not written.
 * Launches three kernels (count, scan, scatter+gather); no atomics on data.
 */
MOE_API moe_status moe_route_sort(const int32_t *topk_ids, int32_t T, int32_t k, int32_t E,
                          int32_t *group_sizes, int32_t *group_offsets, int32_t *sorted_slot,
                          int32_t *slot_to_row, const uint16_t *x, int32_t hidden,
                          uint16_t *x_sorted, moe_act_layout x_sorted_layout, void *workspace,
                          size_t workspace_bytes, void *stream);

/* Size of the fixed scratch array behind moe_route_sort_noalloc (512 KiB). */
#define MOE_ROUTE_SORT_NOALLOC_SCRATCH_BYTES (512u * 1024u)

/*
 * moe_route_sort_noalloc — moe_route_sort for callers that cannot supply a
 * workspace.  The pages have no counterpart of this call; it is an addition of
 * this library.
 *
 * Who needs it: a caller that must not allocate device memory at the point of
 * the call.  Examples are a token-by-token decode loop, where cudaMalloc or
 * cudaFree (directly, or inside a framework's caching allocator when its pool
 * runs dry) may synchronise the device and stall every stream, and an operator
 * with a fixed signature that has no argument through which a scratch buffer
 * could be passed.  This call therefore allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating call into CUDA libraries or into torch.  The counting
 * sort's scratch (per-chunk expert totals and per-slot ranks) and its status
 * word sit in one array of static device storage inside the library, one copy
 * per device.
 *
 * Arguments are those of moe_route_sort without workspace and workspace_bytes,
 * and the results are identical to it on the same inputs.
 *
 * Capacity: the array holds MOE_ROUTE_SORT_NOALLOC_SCRATCH_BYTES of scratch.
 * When moe_workspace_bytes(T, k, E) - 256 exceeds it, the call returns
 * MOE_ERR_CAPACITY and enqueues nothing.  For scale: T*k = 65536 routed slots
 * with E = 256 need 320 KiB.
 *
 * First call: on each device, the first call looks up the device address of
 * the array (cudaGetSymbolAddress, with that device current) and sets a kernel
 * attribute; the lookup may make the driver load the library's device code.
 * Make one call on every device before any stream capture begins.  The address
 * is kept with the CUDA context it was looked up in; when the calling thread's
 * current context differs (another thread before its first CUDA call, or a new
 * primary context after cudaDeviceReset), the call looks the address up again.
 *
 * Overlap: every call on a device shares the one array.  Two calls whose kernels
 * can run at the same time (streams with no ordering between them, or host
 * threads launching concurrently) race on it and produce wrong results; the
 * caller must order them, e.g. by issuing them on one stream.
 *
 * Zeroing: the chunk totals and ranks are written in full before they are
 * read, so they need no clearing.  The status word must start at zero; each
 * call clears it with a stream-ordered cudaMemsetAsync before its kernels.
 *
 * Errors: host checks as in moe_route_sort, then the capacity check.  No
 * status word is exposed: a slot whose id lies outside [0, E) is left out of
 * every band, so group_offsets[E] < T*k tells the caller that it happened.
 */
MOE_API moe_status moe_route_sort_noalloc(const int32_t *topk_ids, int32_t T, int32_t k,
                                          int32_t E, int32_t *group_sizes,
                                          int32_t *group_offsets, int32_t *sorted_slot,
                                          int32_t *slot_to_row, const uint16_t *x,
                                          int32_t hidden, uint16_t *x_sorted,
                                          moe_act_layout x_sorted_layout, void *stream);

/*
 * moe_mxfp4_grouped_gemm — W4A16 grouped matmul over expert row bands ([TPU]
 * section 1: the grouped-matmul loop nest with the 4-bit decode step, and the
 * block scale of every 32 weights applied to the decoded tile before the matmul).
 *
 *   out[r, n] = sum_k act[r, k] * e2m1(code[e, n, k]) * 2^(scale[e, n, k/32] - 127)
 *
 * for every row r of band e (bands laid out in expert order by group_sizes).
 *
 *  act          device bf16 [rows, K], 16-byte aligned; rows >= 0.
 *  act_layout   order of act's reduction dimension (row-major or K8-interleaved).
 *  K            reduction length, multiple of 32 (one E8M0 scale per 32).
 *  codes        device uint8 [E, N, K/2], 16-byte aligned: two e2m1 nibbles per
 *               byte, element 2j in bits 0-3; nibble bit 3 = sign, bits 2-1 =
 *               exponent, bit 0 = mantissa; code 0x8 reads as +0.
 *  scales       device uint8 [E, N, K/32]: E8M0 bytes (127 = 1.0); 0..252
 *               supported, 253..255 set MOE_ERR_DATA and produce NaN.
 *  group_sizes  device int32 [E]: rows per expert, >= 0, summing to rows
 *               (else MOE_ERR_DATA and no output is written).
 *  E            1..1024 experts.  N >= 1 output columns.
 *  out          device [rows, N], f32 (4-byte aligned) or bf16 (RNE).
 *  workspace    device, >= 256 bytes (status word).
 * Each call enqueues two kernel launches: bands of 1..32 rows (streamed
 * weights, split accumulators) and bands of more rows (128- or 256-token
 * work items); a launch whose class has no band exits at once.  The second
 * is a programmatic dependent launch that may overlap the first (the two
 * read the same inputs and write disjoint rows).  Work enqueued after the
 * call in the ordinary way waits for both.  A kernel enqueued right after it
 * with programmatic stream serialization must not rely on griddepcontrol.wait
 * (cudaGridDependencySynchronize) alone to see the rows of the first launch:
 * that waits for the second launch only.
 * Every weight is decoded exactly to bf16.  With scale bytes >= 2 every
 * nonzero weight is a normal bf16 number, its products with bf16 activations
 * are exact in f32, and results differ from an exact sum only by f32
 * accumulation order.  Scale bytes 0 and 1 make the smallest weights bf16
 * subnormals (below 2^-126), which the tensor core may read as zero; for
 * those blocks only the accumulation bound, not exactness, is claimed.
 * Empty experts launch no work and their weights are never read.
 */
MOE_API moe_status moe_mxfp4_grouped_gemm(const uint16_t *act, moe_act_layout act_layout,
                                  int64_t rows, int32_t K,
                                  const uint8_t *codes, const uint8_t *scales,
                                  const int32_t *group_sizes, int32_t E, int32_t N, void *out,
                                  moe_dtype out_dtype, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * moe_mxfp4_grouped_gemm_block — moe_mxfp4_grouped_gemm with a choice of how
 * many consecutive k share one E8M0 scale ([TPU] section 1: the kernel is
 * measured "with block 32" and "with block 512"; read here as the scale block).
 *
 *   out[r, n] = sum_k act[r, k] * e2m1(code[e, n, k]) * 2^(scale[e, n, k/scale_block] - 127)
 *
 *  scale_block  32 (MXFP4 proper: identical to moe_mxfp4_grouped_gemm) or 512.
 *  K            a multiple of scale_block.
 *  scales       device uint8 [E, N, K/scale_block].
 * Everything else as for moe_mxfp4_grouped_gemm.  With scale_block 512 the
 * scale bytes are read by the converter threads (a row of K/512 bytes is too
 * short for a TMA box); the tensor-core path is the same.
 */
MOE_API moe_status moe_mxfp4_grouped_gemm_block(const uint16_t *act, moe_act_layout act_layout,
                                                int64_t rows, int32_t K, int32_t scale_block,
                                                const uint8_t *codes, const uint8_t *scales,
                                                const int32_t *group_sizes, int32_t E, int32_t N,
                                                void *out, moe_dtype out_dtype, void *workspace,
                                                size_t workspace_bytes, void *stream);

/*
 * moe_mxfp4_grouped_gemm_swiglu — the w13 grouped matmul with the SwiGLU
 * activation in its epilogue ([TPU] section 1: the w13 matmul and the
 * fused-activation sweep that brought the 4,096-token w13 from 10.1 ms to
 * 3.2 ms; [NVFP4]: w1 and w3 fused into one weight tensor, gate rows first).
 *
 *   y[r, n] = sum_k act[r, k] * e2m1(code[e, n, k]) * 2^(scale[e, n, k/32] - 127)
 *   h[r, i] = silu(y[r, i]) * y[r, I + i],   silu(g) = g / (1 + e^-g)
 *
 * for every row r of band e, i < I.  y is formed in f32 exactly as
 * moe_mxfp4_grouped_gemm forms it (same MMA order), h is computed in f32 as
 * moe_swiglu computes it and rounded once to bf16: the output equals
 * moe_swiglu(moe_mxfp4_grouped_gemm(...) in f32) bit for bit, and y is never
 * written to memory.
 *
 * Arguments as for moe_mxfp4_grouped_gemm, except:
 *  codes / scales  [E, 2*I, K/2] / [E, 2*I, K/32]: rows [0, I) gate, [I, 2I) up.
 *  I               output columns of h, a positive multiple of 16.
 *  h               device bf16 [rows, I] out, 2-byte aligned.
 *  h_layout        order of h's columns (K8-interleaved needs I % 8 == 0), so h
 *                  can feed the w2 grouped matmul directly.
 * Each 128-row weight tile holds 64 gate rows and the matching 64 up rows (an
 * interleave in groups of 16 done by the tile loads, one 5-D TMA box per
 * stage; the weights in memory keep the [gate | up] layout).
 */
MOE_API moe_status moe_mxfp4_grouped_gemm_swiglu(const uint16_t *act, moe_act_layout act_layout,
                                                 int64_t rows, int32_t K, const uint8_t *codes,
                                                 const uint8_t *scales, const int32_t *group_sizes,
                                                 int32_t E, int32_t I, uint16_t *h,
                                                 moe_act_layout h_layout, void *workspace,
                                                 size_t workspace_bytes, void *stream);

/*
 * moe_mxfp4_grouped_gemm_swiglu_gather — moe_mxfp4_grouped_gemm_swiglu with the
 * activation permutation fused into the activation load ([TPU] section 1: the
 * activation permutation that the grouped-matmul timings leave out).  Sorted
 * row r (of band e, in the order of moe_route_sort) takes its activations from
 * token row sorted_slot[r] / top_k of x_k8, fetched by four-row TMA gathers, so
 * no [rows, K] copy of the activations is ever written.  Outputs are identical,
 * bit for bit, to moe_mxfp4_grouped_gemm_swiglu on the gathered rows.
 *
 *  x_k8         device bf16 [T, K], K8-interleaved (moe_act_interleave_k8, or
 *               moe_layer_forward's route step), 16-byte aligned.
 *  T, top_k     token rows of x_k8 and routing choices per token.
 *  sorted_slot  device int32 [rows] from moe_route_sort (row -> slot).  An
 *               entry whose token lies outside [0, T) sets MOE_ERR_DATA (the
 *               row then reads the nearest token row; its outputs are wrong).
 *  Other arguments as for moe_mxfp4_grouped_gemm_swiglu; h is written in the
 *  sorted row order.
 */
MOE_API moe_status moe_mxfp4_grouped_gemm_swiglu_gather(const uint16_t *x_k8, int32_t T,
                                                        int32_t top_k, const int32_t *sorted_slot,
                                                        int64_t rows, int32_t K,
                                                        const uint8_t *codes, const uint8_t *scales,
                                                        const int32_t *group_sizes, int32_t E,
                                                        int32_t I, uint16_t *h,
                                                        moe_act_layout h_layout, void *workspace,
                                                        size_t workspace_bytes, void *stream);

/*
 * moe_mxfp4_grouped_gemm_scatter — moe_mxfp4_grouped_gemm writing sorted row r
 * of the result to row out_row[r] of `out` ([TPU] section 1: the permutation
 * back to slot order, here fused into the epilogue).  With out_row =
 * sorted_slot from moe_route_sort, out is in slot order (row t*k + j for token
 * t's j-th choice) and moe_combine_slots reads it without an index.
 *
 *  out_row      device int32 [rows].  An entry outside [0, rows) is skipped and
 *               sets MOE_ERR_DATA; rows of `out` that no entry names are not
 *               written.
 *  Other arguments as for moe_mxfp4_grouped_gemm.
 */
MOE_API moe_status moe_mxfp4_grouped_gemm_scatter(const uint16_t *act, moe_act_layout act_layout,
                                                  int64_t rows, int32_t K, const uint8_t *codes,
                                                  const uint8_t *scales, const int32_t *group_sizes,
                                                  int32_t E, int32_t N, const int32_t *out_row,
                                                  void *out, moe_dtype out_dtype, void *workspace,
                                                  size_t workspace_bytes, void *stream);

/*
 * moe_nvfp4_grouped_gemm — the same grouped matmul with NVFP4 weights ([TPU]
 * section 1: the NVFP4 kernel that decodes e2m1 weights and per-16 E4M3 scales;
 * [NVFP4] "The lossless weight cast": per-16 E4M3 block scales under a
 * per-tensor f32 weight_scale_2).
 *
 *   out[r, n] = sum_k act[r, k] * e2m1(code[e, n, k]) * e4m3(scales16[e, n, k/16])
 *                              * weight_scale_2[e]
 *
 * for every row r of band e.  Arguments as for moe_mxfp4_grouped_gemm, except:
 *  scales16        device uint8 [E, N, K/16]: E4M3 bytes (sign, 4 exponent bits
 *                  with bias 7, 3 mantissa bits).  0x7F and 0xFF (NaN) set
 *                  MOE_ERR_DATA and produce NaN.
 *  weight_scale_2  device f32 [E], 4-byte aligned.
 *  K               multiple of 32.
 * Each weight e2m1 * E4M3 * 2^-9 is exact in bf16, its products with bf16
 * activations are exact in f32, and the f32 sums are multiplied by 2^9 *
 * weight_scale_2 once per output.  Weights cast losslessly from MXFP4
 * (moe_mxfp4_to_nvfp4) therefore give exactly the outputs of
 * moe_mxfp4_grouped_gemm on the original weights.
 */
MOE_API moe_status moe_nvfp4_grouped_gemm(const uint16_t *act, moe_act_layout act_layout,
                                          int64_t rows, int32_t K, const uint8_t *codes,
                                          const uint8_t *scales16, const float *weight_scale_2,
                                          const int32_t *group_sizes, int32_t E, int32_t N,
                                          void *out, moe_dtype out_dtype, void *workspace,
                                          size_t workspace_bytes, void *stream);

/*
 * moe_swiglu — gate/up activation on the fused w13 output ([TPU] section 1,
 * where the activation is timed apart from the grouped matmuls; [NVFP4]: w1
 * and w3 fused into the first GEMM).
 *
 *   h[r, i] = silu(gu[r, i]) * gu[r, I + i],  silu(g) = g / (1 + e^-g),
 * computed in f32 and rounded once to bf16 (nearest-even).
 *
 *  gu     device [rows, 2*I], f32 or bf16 (in_dtype), 16-byte aligned.
 *  h      device bf16 [rows, I] out, 16-byte aligned.
 *  h_layout  order of h's columns (K8-interleaved needs I % 8 == 0), so that h
 *         can feed the next grouped GEMM directly.
 */
MOE_API moe_status moe_swiglu(const void *gu, moe_dtype in_dtype, int64_t rows, int32_t I, uint16_t *h,
                      moe_act_layout h_layout, void *stream);

/*
 * moe_combine — deterministic top-k weighted unpermute ([Pocket]: expert
 * reduction without atomicAdd).
 *
 *   out[t, n] = sum_{j = 0..k-1} topk_w[t, j] * y[slot_to_row[t*k + j], n]
 *
 * summed as an f32 fused-multiply-add chain in ascending j, so results are
 * bitwise reproducible run to run.
 *
 *  y            device f32 [T*k, N], 16-byte aligned.
 *  slot_to_row  device int32 [T*k] (from moe_route_sort).  An entry outside
 *               [0, T*k) (moe_route_sort writes -1 for an id out of range)
 *               adds nothing: y is never read outside its T*k rows.
 *  topk_w       device f32 [T, k].
 *  out          device [T, N], f32 or bf16.
 */
MOE_API moe_status moe_combine(const float *y, const int32_t *slot_to_row, const float *topk_w,
                       int32_t T, int32_t k, int32_t N, void *out, moe_dtype out_dtype,
                       void *stream);

/*
 * moe_combine_slots — moe_combine with y in slot order:
 *
 *   out[t, n] = sum_{j = 0..k-1} topk_w[t, j] * y[t*k + j, n]
 *
 * over the slots whose slot_to_row entry lies in [0, T*k) (moe_route_sort
 * writes -1 for an id out of range; such a slot adds nothing and its y row is
 * never read).  Same f32 FMA chain in ascending j as moe_combine, so for y
 * permuted to slot order the results are identical bit for bit.
 *  y            device f32 [T*k, N] in slot order, 16-byte aligned.
 *  Other arguments as for moe_combine.
 */
MOE_API moe_status moe_combine_slots(const float *y, const int32_t *slot_to_row, const float *topk_w,
                                     int32_t T, int32_t k, int32_t N, void *out, moe_dtype out_dtype,
                                     void *stream);

/*
 * moe_act_interleave_k8 — activations in the K8-interleaved order the grouped
 * GEMMs consume: within every 8 consecutive bf16 of a row, element e moves to
 * position 2e (e < 4) or 2(e - 4) + 1.
 *  x, x_k8      device bf16 [rows, hidden], 16-byte aligned, hidden % 8 == 0.
 */
MOE_API moe_status moe_act_interleave_k8(const uint16_t *x, int64_t rows, int32_t hidden,
                                         uint16_t *x_k8, void *stream);

/*
 * moe_layer_forward — the whole routed-expert path in one call:
 * route_sort (with gather) -> w13 grouped GEMM with SwiGLU in its epilogue
 * (moe_mxfp4_grouped_gemm_swiglu) -> w2 grouped GEMM -> combine, each stage as
 * described above, all on `stream` (eight kernel launches).  x_sorted and h are
 * written in the K8-interleaved order; the f32 gate/up product is never
 * written.
 *
 *  x            device bf16 [T, hidden]; topk_ids int32 [T, k]; topk_w f32 [T, k].
 *  w13_codes/scales  [E, 2*inter, hidden/2] / [E, 2*inter, hidden/32]
 *               (output columns [0, inter) gate, [inter, 2*inter) up).
 *  w2_codes/scales   [E, hidden, inter/2] / [E, hidden, inter/32].
 *  out          device f32 [T, hidden].
 *  Caller-owned intermediates (device): group_sizes int32 [E], group_offsets
 *  int32 [E+1], sorted_slot / slot_to_row int32 [T*k], x_sorted bf16
 *  [T*k, hidden], h bf16 [T*k, inter], y2 f32 [T*k, hidden], workspace >=
 *  moe_workspace_bytes(T, k, E).
 * hidden and inter must be multiples of 32.
 */
MOE_API moe_status moe_layer_forward(const uint16_t *x, const int32_t *topk_ids, const float *topk_w,
                             int32_t T, int32_t k, int32_t E, int32_t hidden, int32_t inter,
                             const uint8_t *w13_codes, const uint8_t *w13_scales,
                             const uint8_t *w2_codes, const uint8_t *w2_scales, float *out,
                             int32_t *group_sizes, int32_t *group_offsets, int32_t *sorted_slot,
                             int32_t *slot_to_row, uint16_t *x_sorted, uint16_t *h, float *y2,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * moe_set_gemm_pairing — how the grouped GEMMs (MXFP4 plain, block 512 and
 * fused SwiGLU, and NVFP4) run bands of more than 32 rows; process-wide, for
 * every later call.
 *  MOE_PAIRING_AUTO  CTA pairs when K8 activations, an even number of column
 *                    tiles (128 output rows, or 64 h columns, each) and rows
 *                    >= 64 * E (the bands average at least 64 rows).
 *  MOE_PAIRING_OFF   one CTA per work item.
 *  MOE_PAIRING_ON    CTA pairs whenever K8 activations and an even tile count.
 * In a CTA pair (a cluster of two CTAs on two SMs) each work item is a 256-row
 * weight tile, 128 rows decoded by each CTA, and up to 256 token rows, half
 * loaded by each CTA; the even CTA issues M = 256 tensor-core MMAs over both.
 * Each SM thus loads half of every activation tile.  Results are identical
 * either way (same products, same accumulation order).
 */
typedef enum { MOE_PAIRING_AUTO = 0, MOE_PAIRING_OFF = 1, MOE_PAIRING_ON = 2 } moe_pairing;
MOE_API moe_status moe_set_gemm_pairing(int32_t mode);

/*
 * moe_mxfp4_decode_expert — debug view of the GEMM's weight decode: writes
 * expert e's weights e2m1(code) * 2^(scale - 127) as bf16 [N, K], produced by
 * the same device routine the GEMM's converter warps run.  Used to check the
 * decode bit for bit.  Same code/scale layout and status rules as the GEMM.
 */
MOE_API moe_status moe_mxfp4_decode_expert(const uint8_t *codes, const uint8_t *scales, int32_t E,
                                   int32_t N, int32_t K, int32_t e, uint16_t *out,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device workspace needed by moe_mxfp4_to_nvfp4 for E experts: the
 * status word plus one 32-bit scratch word per expert. */
MOE_API size_t moe_nvfp4_cast_workspace_bytes(int32_t E);

/*
 * moe_mxfp4_to_nvfp4 — lossless cast of MXFP4 weight scales to NVFP4's two
 * scale levels ([NVFP4] "The lossless weight cast").  The e2m1 codes are
 * shared by both formats and are not touched; only the scales change.
 *
 * For each expert e, over its whole scale tensor (so the w1 and w3 rows of a
 * fused w13 tensor share one per-tensor scale), with k_max = max(s) - 127:
 *   weight_scale_2[e]          = 2^(k_max - 8)                 (f32, exact)
 *   e4m3_scales[e, n, 2b], [2b+1] = 2^(s[e, n, b] - 127 - k_max + 8) (E4M3)
 * so that E4M3 scale x weight_scale_2 = 2^(s - 127) for every 16-element half
 * of every 32-block: each weight dequantizes to exactly its MXFP4 value.  E4M3
 * holds the powers of two 2^-9..2^8, so a block whose scale lies more than 17
 * binades below the expert's largest has no exact E4M3 scale: its two bytes
 * are written as 0 and it is counted in out_of_range[e] (the exactness audit;
 * 0 means the cast is lossless for that expert).
 *
 *  scales          device uint8 [E, N, K/32]: E8M0 bytes (127 = 1.0).  Byte
 *                  255 (NaN) sets MOE_ERR_DATA; the outputs are then
 *                  unspecified.
 *  E, N, K         experts (1..65535), rows per expert (>= 1), reduction
 *                  length (multiple of 32).
 *  e4m3_scales     device uint8 [E, N, K/16] out: E4M3 bytes (sign 0, 4
 *                  exponent bits with bias 7, 3 mantissa bits).
 *  weight_scale_2  device f32 [E] out.
 *  out_of_range    device uint64 [E] out: blocks written as 0 (cleared by the
 *                  call before counting).
 *  workspace       device, >= moe_nvfp4_cast_workspace_bytes(E) bytes,
 *                  16-byte aligned; its status word as for every call.
 * Launches one kernel when each expert's scale tensor (N * K/32 bytes) is a
 * multiple of 16 bytes and at most 512 KiB and both byte buffers are 16-byte
 * aligned: persistent clusters of up to 8 CTAs (64 KiB of an expert each) read
 * the scales once.  Otherwise two kernels (per-expert maximum into the
 * workspace, then the conversion).  A bulk copy or a message between the CTAs
 * of a cluster that does not arrive within 2 s records MOE_ERR_TIMEOUT.
 * Results are exact integers, identical from run to run.
 */
MOE_API moe_status moe_mxfp4_to_nvfp4(const uint8_t *scales, int32_t E, int32_t N, int32_t K,
                                      uint8_t *e4m3_scales, float *weight_scale_2,
                                      uint64_t *out_of_range, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * moe_debug_bounded_wait — failure-detection self-test.  Launches one block
 * that waits on a shared-memory barrier nothing will ever complete, using the
 * same bounded wait as the GEMM pipeline with a limit of `limit_ns`
 * nanoseconds (1e3..5e9).  The wait gives up, records MOE_ERR_TIMEOUT in the
 * status word and the kernel returns; the CUDA context stays usable.
 */
MOE_API moe_status moe_debug_bounded_wait(uint64_t limit_ns, void *workspace, size_t workspace_bytes,
                                  void *stream);

/* Number of kernel launches the last successful call on this host thread
 * enqueued (for launch accounting in benchmarks). */
MOE_API int32_t moe_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_MXFP4_H */
