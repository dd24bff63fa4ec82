// MXFP4 and NVFP4 (W4A16) grouped GEMM over expert-sorted row bands, sm_103a.
//
// NVFP4 ("DeepSeek-V4-Flash-0731-NVFP4", "The lossless weight cast": per-16
// E4M3 block scales under a per-tensor weight_scale_2) runs the same kernel
// body (grouped_gemm_nvfp4_kernel): every 16 codes take the constant
// bf16(E4M3 * 2^117) from a 256-entry shared-memory table, so each decoded
// weight e2m1 * E4M3 * 2^-9 is still one exact bf16 FMA, and the epilogue
// multiplies the f32 sums by 2^9 * weight_scale_2.
//
// What it computes ("Running DeepSeek V4 Flash on TPU v6", section 1, the
// grouped-matmul loop nest with the decode step): for every expert e with a
// non-empty band of rows, out[r, n] = sum_k act[r, k] * w_e[n, k], where
// w_e[n, k] = e2m1(code) * 2^(scale - 127) is decoded exactly to bf16 before
// the matmul, bf16 products are exact in f32 and accumulate in f32.
//
// How (GB300 design, not the page's TPU design):
//  * Swap-AB: the decoded weight tile (128 output columns n x K) is the MMA's A
//    operand, held in tensor memory; the band's token rows are the B operand
//    in shared memory (MMA N = 16..256).  Decode-sized bands thus fill the
//    128-wide tensor-core dimension with weights, not with padding.
//  * A ring of code stages in shared memory, filled by TMA: each holds the
//    codes of 128 rows x 256 k (128-byte swizzle), the block-scale bytes when
//    K % 512 == 0, and for narrow bands the band's activation tile of the same
//    256 k, so activations arrive as early as the codes.  Wider bands take
//    their activations through 64-k slots of their own.
//  * Four converter warpgroups decode in pairs on alternate code stages: each
//    warpgroup takes one 128-k half; a thread reads the 64 code bytes of its
//    weight row, decodes them to bf16 pairs on the ALU and FMA pipes and
//    writes them into the warpgroup's two tensor-memory A slots (tcgen05.st).
//  * Split mode (every band <= 32 rows): two issuer warps, each issuing two
//    adjacent 64-k sub-stages of every code stage into its own K-partial
//    accumulator; the epilogue adds the partials in a fixed order (one issuer
//    thread issues a small MMA only about every 50 cycles, so the work is
//    shared).  Single mode (bands up to 128 rows): the two issuers split the
//    token columns of one accumulator and take four stages per barrier probe;
//    accumulators are double-buffered so the epilogue of one work item (done
//    by the converter warps) overlaps the next item.  Wide mode (a band over
//    128 rows, K8 activations): 256-token items, so each decoded weight feeds
//    twice the MMA work; one issuer, one 256-column accumulator, five
//    activation slots.
//  * Fused SwiGLU (w13): a weight tile holds 64 gate rows and their 64 up
//    rows, so the epilogue forms h = silu(g) * u and y13 is never stored.
//  * Persistent CTAs (one per SM) walk a static list of work items (expert,
//    token chunk, column tile) built on the device from group_sizes; empty
//    experts contribute no items and their weights are never read.
//  * Every wait is bounded (no unbounded barrier inside the pipeline); on
//    timeout the kernel records MOE_ERR_TIMEOUT, drains its own copies and
//    MMAs, frees tensor memory and returns.
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "device_common.cuh"
#include "launch.h"
#include "mxfp4_decode.cuh"

namespace moe {
namespace gemm {

constexpr int kIssuerWarps = 2;               // warps 0..1: MMA issuers (one elected lane each)
constexpr int kSingleIssuers = 2;             // single mode: issuers splitting the token columns
// Wide mode: one issuer issues each stage as MMAs of N = the item's tokens
// (up to 256), half the instructions of two issuers splitting the columns.
constexpr int kWideIssuers = 1;
constexpr int kConvWG = 4;                    // converter warpgroups: warps 2..17
constexpr int kConvWarp0 = kIssuerWarps;
constexpr int kActWarp = kConvWarp0 + 4 * kConvWG;    // warp 18: activation producer
constexpr int kCodeWarp = kActWarp + 1;               // warp 19: code producer
constexpr int kThreads = 32 * (kCodeWarp + 1);        // 640
constexpr int kBN = 128;                      // output columns per tile (MMA M)
constexpr int kMaxNT = 128;                   // tokens per work item (MMA N)
constexpr int kWideNT = 256;                  // wide mode: tokens per work item
// Wide mode: activation slots (32 KB each).  Five leave room for two code
// stages (the ring depth must be even), one per converter pair: the
// converters run far ahead of the tensor core, while the activation tiles
// (re-read from L2 for every column tile) need the deeper prefetch.
constexpr int kWideActSlots = 5;
// Pair mode: activation slots of up to 16 KB (a CTA's half of 256 tokens); ten
// leave room for two code stages, one per converter pair (measured best).
constexpr int kPairActSlots = 10;
constexpr int kStageK = 64;                   // K per decode / MMA stage
constexpr int kSlots = 8;                     // A slots in TMEM (+ activation slots in smem)
constexpr int kSlotsMax = 12;                 // bands <= 16 rows: three A slots per warpgroup
constexpr int kCodeK = 256;                   // K per code stage (4 decode stages)
constexpr int kCodeStageBytes = kBN * kCodeK / 2;         // 16 KB
constexpr int kCodeStagesMax = 12;
constexpr int kScaleTileBytes = 128 * 16;     // scale bytes of two code stages (512 k) x 128 rows
constexpr int kRingBytes = 214 * 1024;        // code ring + activation tiles
constexpr int kItemCache = 128;               // work items of a CTA kept decoded in shared memory
constexpr int kTmemCols = 512;
constexpr int kAccCols = 128;                 // per accumulator buffer
constexpr int kACol0 = 2 * kAccCols;          // A slots after the two accumulator buffers
constexpr int kAColsPerSlot = kStageK / 2;    // bf16 pairs: 32 columns
constexpr int kPartCols = 32;                 // split mode: columns of one K-partial
constexpr int kMaxE = 1024;

constexpr int kOffCode = 0;
constexpr int kOffRowOff = kOffCode + kRingBytes;
constexpr int kOffItemOff = kOffRowOff + (kMaxE + 1) * 4;
constexpr int kOffBars = (kOffItemOff + (kMaxE + 1) * 4 + 7) & ~7;
constexpr int kNumBars = 2 * kCodeStagesMax + 4 * kSlotsMax + 2 * 2 + kIssuerWarps;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kOffItems = (kOffMisc + 64 + 15) & ~15;     // int4 per cached work item (16-aligned)
constexpr int kSmemBytes = kOffItems + kItemCache * 16 + 1024;   // + alignment slack

// NVFP4: a 256-entry table of per-16 scale constants after the item table.
constexpr int kOffNvTab = kOffItems + kItemCache * 16;
constexpr int kSmemBytesNv = kOffNvTab + 256 * 4 + 1024;

static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kSmemBytesNv <= 232448, "shared memory budget (NVFP4)");
static_assert(kOffItems % 16 == 0, "the item table holds int4 entries");
static_assert(kCodeStageBytes % 1024 == 0, "ring slots keep the 1024-byte swizzle alignment");
static_assert(kOffBars % 8 == 0, "barrier alignment");
static_assert(kACol0 + kSlots * kAColsPerSlot <= kTmemCols, "TMEM budget");
static_assert(kSlots == 2 * kConvWG, "each warpgroup alternates between two A slots");
static_assert(kConvWG * kPartCols <= kAccCols, "split-mode partials fit one buffer");
static_assert(2 * kConvWG * (kPartCols / 2) + kSlotsMax * kAColsPerSlot <= kTmemCols,
              "narrow layout: 16-column partials, twelve A slots");
static_assert(kCodeK / kStageK == kConvWG, "one code stage = one decode stage per warpgroup");

struct Params {
    const uint8_t *scales;
    const int32_t *group_sizes;
    void *out;
    int *status;
    int rows, K, N, E;
    int out_bf16;
    int n_tiles;       // ceil(N / 128)
    int k_stages;      // 64-k stages per item: 4 * ceil(K / 256)
    int scale_row;     // scale bytes a weight row: K / block (MXFP4), K / 16 (NVFP4)
    int k_blocks;      // K / 32: 32-k blocks a weight row
    int scale_shift;   // MXFP4: log2(block / 32); 32-k block b takes scale byte b >> scale_shift
    int scale_vec2;    // scale rows 2-byte aligned: load a stage's 2 scale bytes at once
    int scale_full;    // scale_vec2 and K % 256 == 0: every stage has both scale bytes
    int scale_tma;     // K % 512 == 0, 16-byte aligned scales: scale tiles ride in the ring
    int act_k8;        // activations already in the K8-interleaved order
    int act3d;         // K % 256 == 0: one 3-D box fetches a band's 256-k activation tile
    // Fused SwiGLU (w13 with N = 2 * I rows, gate rows [0, I), up rows [I, 2I)):
    // a tile holds 64 gate rows and the 64 matching up rows, interleaved in
    // groups of 16 (tile row 32q + i: gate row n0 + 16q + i; 32q + 16 + i: up
    // row I + n0 + 16q + i), and the epilogue writes h = silu(g) * u as bf16
    // [rows, I] (K8-interleaved when h_k8).  n_tiles = ceil(I / 64) then.
    int swiglu;
    int I;
    int h_k8;
    int allow_wide;    // K8 activations: bands over 128 rows take 256-token items
    // Band class of this launch: only experts with band_lo <= rows <= band_hi
    // get work items (row offsets still count every expert).  A grouped GEMM
    // is two launches, bands up to 32 rows (split mode, weight streaming) and
    // longer ones (single or wide mode), so a mix of short and long bands
    // runs each in the mode made for it.
    int band_lo, band_hi;
    // Activation gather (the routing permutation fused into the activation
    // load; the kGather instantiation): sorted row r reads row gather_slot[r] /
    // gather_k of a [act_rows, K] activation tensor, four rows per TMA (tm_act
    // and tm_act64 are then one-row gather maps).
    const int32_t *gather_slot;
    int gather_k;
    int act_rows;
    // Output scatter (the kScatter instantiation): sorted row r is written to
    // row out_row[r] of the output; an entry outside [0, rows) is skipped and
    // recorded as MOE_ERR_DATA.
    const int32_t *out_row;
    uint64_t wait_limit_ns;
};

// Row maps of a launch: none, the activation gather, or the output scatter.
// Each is its own kernel instantiation, so the plain kernels carry no trace of
// the other two.
enum RowMap { kMapNone = 0, kMapGather = 1, kMapScatter = 2 };

// Activation row of sorted row r under the gather: gather_slot[r] / gather_k,
// clamped into [0, act_rows) (a row outside records MOE_ERR_DATA).
__device__ __forceinline__ int gather_row(const Params &p, int r) {
    const int a = __ldg(p.gather_slot + r) / p.gather_k;
    if (a < 0 || a >= p.act_rows) {
        set_status(p.status, MOE_ERR_DATA);
        return a < 0 ? 0 : p.act_rows - 1;
    }
    return a;
}

// Scatter: output row of sorted row r, or -1 (recorded) when out of range.
__device__ __forceinline__ int scatter_row(const Params &p, int r) {
    const int o = __ldg(p.out_row + r);
    if (o < 0 || o >= p.rows) {
        set_status(p.status, MOE_ERR_DATA);
        return -1;
    }
    return o;
}

struct Item {
    int e, row0, nvalid, nt, n0;
};

// Work item j -> (expert, token chunk, column tile); ioff/roff in shared
// memory.  chunk: tokens per item (128, or 256 in wide mode).  n0 is the
// first output column of the tile: weight row n0 (plain) or h column n0 (fused
// SwiGLU, 64 columns a tile).
__device__ __forceinline__ Item decode_item(int j, const int *roff, const int *ioff, int E,
                                            int n_tiles, int chunk, int tile_cols) {
    int lo = 0, hi = E - 1;   // last e with ioff[e] <= j (its band is non-empty)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ioff[mid] <= j) lo = mid; else hi = mid - 1;
    }
    Item it;
    it.e = lo;
    const int r = j - ioff[lo];
    const int ch = r / n_tiles;
    it.n0 = (r - ch * n_tiles) * tile_cols;
    const int t0 = ch * chunk;
    const int rem = roff[lo + 1] - roff[lo] - t0;
    it.nvalid = rem < chunk ? rem : chunk;
    it.nt = (it.nvalid + 15) & ~15;
    it.row0 = roff[lo] + t0;
    return it;
}

// Fused SwiGLU tile layout: tile row (TMEM lane) -> offset of its weight row
// from n0 (up rows carry + I), and whether it is an up row.
__device__ __forceinline__ int swiglu_row_offset(int row) {
    return 16 * (row >> 5) + (row & 15);
}
__device__ __forceinline__ bool swiglu_row_is_up(int row) { return (row & 16) != 0; }

// Column j of h in the K8-interleaved order: within each 8, element e is
// stored at position 2e (e < 4) or 2(e - 4) + 1.
__device__ __forceinline__ int k8_position(int j) {
    return (j & ~7) | ((j & 3) << 1) | ((j >> 2) & 1);
}

// Position in a ring of `n` mbarrier-guarded slots: slot index and the parity
// of the phase the current use waits for.  Advancing flips the parity on wrap.
struct Ring {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void next(uint32_t n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// Epilogue of one work item for converter warpgroup `wg`: the warpgroup writes
// its quarter of the item's token columns.  In split mode the two K-partials
// are added in a fixed order (deterministic); f32 or bf16 output.  Fused
// SwiGLU: lanes l and l ^ 16 of a warp hold the gate and up sums of the same
// output column, so one shuffle pairs them; lanes 0-15 finish token c, lanes
// 16-31 token c + 1, and h is written as bf16.
// kScatter: token t of the item goes to output row out_row[row0 + t]; lane l
// holds that row for column wg * qc + l (qc <= 32) and shuffles it out.
template <bool kNv, bool kScatter>
__device__ __forceinline__ void store_item(const Params &p, const Item &it, uint32_t acc_base,
                                           int wg, int row, bool split, uint32_t part_cols,
                                           float tensor_scale) {
    const int qc = it.nt >> 2;                 // columns per warpgroup (multiple of 4)
    const bool up_lane = swiglu_row_is_up(row);
    const int n = p.swiglu ? it.n0 + swiglu_row_offset(row) : it.n0 + row;
    int my_orow = -1;
    if constexpr (kScatter) {
        const int t = wg * qc + (threadIdx.x & 31);
        if ((threadIdx.x & 31) < qc && t < it.nvalid) my_orow = scatter_row(p, it.row0 + t);
    }
    for (int c = wg * qc; c < (wg + 1) * qc; c += 4) {
        uint32_t v[4];
        __syncwarp();
        tmem_ld4(acc_base + c, v);
        if (split) {
            uint32_t u1[4];
            tmem_ld4(acc_base + part_cols + c, u1);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < 4; ++t)
                v[t] = __float_as_uint(__uint_as_float(v[t]) + __uint_as_float(u1[t]));
        } else {
            tmem_ld_wait();
        }
        float f[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            f[t] = __uint_as_float(v[t]);
            // NVFP4: the decoded weights carry 2^-9 / weight_scale_2 (exact
            // power-of-two scaling); one rounding restores the scale.
            if constexpr (kNv) f[t] = (f[t] * 512.0f) * tensor_scale;
        }
        if (p.swiglu) {
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const float a0 = f[2 * pr], a1 = f[2 * pr + 1];
                const float recv = __shfl_xor_sync(0xffffffffu, up_lane ? a0 : a1, 16);
                const float g = up_lane ? recv : a0;
                const float u = up_lane ? a1 : recv;
                const int tok = c + 2 * pr + (up_lane ? 1 : 0);
                int orow = it.row0 + tok;
                if constexpr (kScatter) orow = __shfl_sync(0xffffffffu, my_orow, tok - wg * qc);
                if (n < p.I && tok < it.nvalid && (!kScatter || orow >= 0)) {
                    const int col = p.h_k8 ? k8_position(n) : n;
                    const size_t off = static_cast<size_t>(orow) * p.I + col;
                    reinterpret_cast<__nv_bfloat16 *>(p.out)[off] =
                        __float2bfloat16_rn(silu_f32(g) * u);
                }
            }
        } else if (kScatter || n < p.N) {     // scatter: every lane takes part in the shuffles
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int tok = c + t;
                int orow = it.row0 + tok;
                if constexpr (kScatter) orow = __shfl_sync(0xffffffffu, my_orow, tok - wg * qc);
                if ((!kScatter || n < p.N) && tok < it.nvalid && (!kScatter || orow >= 0)) {
                    const size_t off = static_cast<size_t>(orow) * p.N + n;
                    if (p.out_bf16)
                        reinterpret_cast<__nv_bfloat16 *>(p.out)[off] = __float2bfloat16_rn(f[t]);
                    else
                        reinterpret_cast<float *>(p.out)[off] = f[t];
                }
            }
        }
    }
}

// Epilogue of one work item in wide mode (one accumulator, up to 64 columns a
// warpgroup): the columns are read 16 at a time (one load, one wait), so at
// most four load latencies are exposed per warp instead of one per four
// columns.  The caller releases the accumulator afterwards.
// kScatter: as in store_item, with up to 64 columns a warpgroup (two rows a lane).
template <bool kNv, bool kScatter>
__device__ __forceinline__ void store_item_wide(const Params &p, const Item &it, uint32_t acc_base,
                                                int wg, int row, float tensor_scale) {
    const int qc = it.nt >> 2;                 // columns of this warpgroup: <= 64, multiple of 4
    const int cb = wg * qc;
    const bool up_lane = swiglu_row_is_up(row);
    const int n = p.swiglu ? it.n0 + swiglu_row_offset(row) : it.n0 + row;
    int orow_lo = -1, orow_hi = -1;            // scatter: rows of columns cb + lane, cb + 32 + lane
    if constexpr (kScatter) {
        const int l = threadIdx.x & 31;
        if (l < qc && cb + l < it.nvalid) orow_lo = scatter_row(p, it.row0 + cb + l);
        if (32 + l < qc && cb + 32 + l < it.nvalid) orow_hi = scatter_row(p, it.row0 + cb + 32 + l);
    }
    // Output row of token column tok (the warp executes it together).
    auto out_row_of = [&](int tok) -> int {
        if constexpr (kScatter) {
            const int rel = tok - cb;
            const int lo = __shfl_sync(0xffffffffu, orow_lo, rel & 31);
            const int hi = __shfl_sync(0xffffffffu, orow_hi, rel & 31);
            return rel < 32 ? lo : hi;
        } else {
            return it.row0 + tok;
        }
    };
    for (int c16 = 0; c16 < qc; c16 += 16) {
        uint32_t v[16];
        __syncwarp();
        tmem_ld16(acc_base + cb + c16, v);
        tmem_ld_wait();
        {
#pragma unroll
            for (int t = 0; t < 16; t += 2) {
                const int col = c16 + t;            // pair (col, col + 1): both < qc or both >= qc
                if (col >= qc) break;
                float a0 = __uint_as_float(v[t]), a1 = __uint_as_float(v[t + 1]);
                if constexpr (kNv) {
                    a0 = (a0 * 512.0f) * tensor_scale;
                    a1 = (a1 * 512.0f) * tensor_scale;
                }
                if (p.swiglu) {
                    const float recv = __shfl_xor_sync(0xffffffffu, up_lane ? a0 : a1, 16);
                    const float g = up_lane ? recv : a0;
                    const float u = up_lane ? a1 : recv;
                    const int tok = cb + col + (up_lane ? 1 : 0);
                    const int orow = out_row_of(tok);
                    if (n < p.I && tok < it.nvalid && (!kScatter || orow >= 0)) {
                        const int hc = p.h_k8 ? k8_position(n) : n;
                        reinterpret_cast<__nv_bfloat16 *>(p.out)[static_cast<size_t>(orow) * p.I + hc] =
                            __float2bfloat16_rn(silu_f32(g) * u);
                    }
                } else if (kScatter || n < p.N) {   // scatter: every lane takes part in the shuffles
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = cb + col + e;
                        const int orow = out_row_of(tok);
                        if ((!kScatter || n < p.N) && tok < it.nvalid && (!kScatter || orow >= 0)) {
                            const size_t off = static_cast<size_t>(orow) * p.N + n;
                            const float val = e ? a1 : a0;
                            if (p.out_bf16)
                                reinterpret_cast<__nv_bfloat16 *>(p.out)[off] = __float2bfloat16_rn(val);
                            else
                                reinterpret_cast<float *>(p.out)[off] = val;
                        }
                    }
                }
            }
        }
    }
}

// bf16 bits of E4M3 byte b times 2^117, in both halves of a bf16x2.  Exact:
// E4M3 has at most four significant bits, and the factor 2^117 keeps every
// finite value normal in bf16 (2^99 .. 448 * 2^117).  Normal bytes move their
// exponent by 110 + 127; subnormals m * 2^-9 become m * 2^108; 0x7F / 0xFF
// (E4M3 NaN) become a bf16 NaN.
__device__ __forceinline__ uint32_t e4m3_scaled_pair(uint32_t b) {
    const uint32_t mag = b & 0x7Fu;
    uint32_t v;
    if (mag == 0x7Fu) v = 0x7FC0u;
    else if (mag >= 8u) v = (mag << 4) + (237u << 7);
    else if (mag == 0u) v = 0u;
    else v = (__float_as_uint(static_cast<float>(mag)) + (108u << 23)) >> 16;
    v |= (b & 0x80u) << 8;
    return v | (v << 16);
}

// 16 codes (two code words) of one NVFP4 block with its scale constant S:
// o[4w + j] = (element 8w + j, element 8w + j + 4) times S, for w = 0, 1.
__device__ __forceinline__ void decode16_scaled(uint32_t c0, uint32_t c1, uint32_t S, uint32_t *o) {
    uint32_t x[4];
    e2m1_pairs_scaled_down(c0, x);
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = bf16x2_fma(x[j], S, 0u);
    e2m1_pairs_scaled_down(c1, x);
#pragma unroll
    for (int j = 0; j < 4; ++j) o[4 + j] = bf16x2_fma(x[j], S, 0u);
}

// The kernel body for both weight formats.  kNv = false: MXFP4 (per-32 E8M0
// scales).  kNv = true: NVFP4 (per-16 E4M3 scales `p.scales`, per-expert f32
// weight_scale_2 `ws2`): each decoded weight is e2m1 * E4M3 * 2^-9, exact in
// bf16, and the epilogue multiplies by 2^9 * weight_scale_2.  kSplit: the
// launch for bands of at most 32 rows (split mode only); otherwise the launch
// for longer bands (single or wide mode).  Separate instantiations keep each
// mode's loops free of the other modes' code.
template <bool kNv, bool kSplit, int kMap, bool kPair = false>
__device__ __forceinline__ void gemm_body(const CUtensorMap &tm_codes, const CUtensorMap &tm_act,
                                          const CUtensorMap &tm_act3, const CUtensorMap &tm_scales,
                                          const CUtensorMap &tm_act64, const Params &p,
                                          const float *ws2) {
    // A programmatic dependent launch that follows may start as this grid's
    // CTAs retire.  Only the second band-class launch of the same GEMM is
    // launched that way; it depends on nothing this grid writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned start, derived from the shared array itself so that the
    // compiler keeps the shared address space (shared loads, not generic ones).
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    int *roff = reinterpret_cast<int *>(smem + kOffRowOff);
    int *ioff = reinterpret_cast<int *>(smem + kOffItemOff);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars);
    uint64_t *code_full = bars;                          // TMA -> converters (+ issuers, split)
    uint64_t *code_empty = code_full + kCodeStagesMax;   // 16 converter warps (+ 4 commits, split)
    // a_full / slot_empty: one barrier per warpgroup, covering its two A slots
    // (the warpgroup fills both in one stage and they are consumed together).
    uint64_t *a_full = code_empty + kCodeStagesMax;      // converters -> issuer (4 warps)
    uint64_t *act_full = a_full + kSlotsMax;             // TMA -> issuer (single mode)
    uint64_t *slot_empty = act_full + kSlotsMax;         // MMA commit -> converters, act producer
    uint64_t *act_empty = slot_empty + kSlotsMax;        // wide mode: MMA commit -> act producer
    uint64_t *acc_full = act_empty + kSlotsMax;          // MMA commits -> epilogue
    uint64_t *acc_empty = acc_full + 2;                  // epilogue (16 warps) -> issuers
    uint64_t *final_bar = acc_empty + 2;                 // one per issuer thread
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
    int *bad_flag = reinterpret_cast<int *>(smem + kOffMisc + 16);
    int *nt_max_slot = reinterpret_cast<int *>(smem + kOffMisc + 24);
    int *chunk_slot = reinterpret_cast<int *>(smem + kOffMisc + 32);
    int4 *item_cache = reinterpret_cast<int4 *>(smem + kOffItems);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int E = p.E;
    // CTA pair (kPair, wide mode only): the two CTAs of a cluster share every
    // work item.  Each takes 128 weight rows of the pair's 256-row tile (tile
    // 2t + rank of pair tile t) and half of the item's token rows; the even CTA
    // issues M = 256 MMAs over both, so each SM loads half of the activations.
    static_assert(!kPair || (!kSplit && kMap == kMapNone), "pair mode: wide bands, no row maps");
    const uint32_t rank = kPair ? cluster_rank() : 0u;
    const int cta = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int n_cta = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int item_tiles = kPair ? p.n_tiles / 2 : p.n_tiles;    // column tiles a work item list has
    // Tensor-core issue in the instantiation's CTA granularity (a kernel uses
    // the single-CTA or the pair forms throughout).  Pair commits arrive on the
    // barrier in both CTAs, except for the issuer's own final barrier.
    auto mma_issue = [](uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (kPair) mma_bf16_ts_pair(d, a, b, id, acc);
        else mma_bf16_ts(d, a, b, id, acc);
    };
    auto mma_commit_all = [](uint64_t *bar) {
        if constexpr (kPair) mma_commit_pair(bar, 3);
        else mma_commit(bar);
    };
    auto mma_commit_own = [](uint64_t *bar) {
        if constexpr (kPair) mma_commit_pair(bar, 1);
        else mma_commit(bar);
    };

    // ---------------------------------------------------------------- prologue
    if (tid == 0) {
        *abort_flag = 0;
        *bad_flag = 0;
    }
    // The group sizes, staged in roff (which the scan below overwrites entry
    // by entry, each after reading it): one load per thread, all in flight at
    // once, instead of the scanning warp's dependent chunks of 32.
    for (int e = tid; e < E; e += kThreads) roff[e] = p.group_sizes[e];
    __syncthreads();
    // Row offsets and work-item offsets: exclusive prefix sums over experts,
    // done by warp 0 in chunks of 32 (E <= 1024); also the widest work item.
    // The running sums are 64-bit and every prefix is checked against rows, so
    // group sizes whose 32-bit sum would wrap around to rows are still caught.
    // A first pass finds the largest band: with one over 128 rows (and K8
    // activations) every work item takes up to 256 tokens (wide mode).
    if (warp == 0) {
        int g_max = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int gs = e < E ? roff[e] : 0;
            if (gs < 0) *bad_flag = 1;
            if (gs >= p.band_lo && gs <= p.band_hi) g_max = max(g_max, gs);
        }
        g_max = __reduce_max_sync(0xffffffffu, g_max);
        const int chunk = (kPair || (p.allow_wide && g_max > kMaxNT)) ? kWideNT : kMaxNT;
        long long run_rows = 0, run_items = 0;
        int nt_max = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int gs = e < E ? roff[e] : 0;
            const int g = gs > 0 ? gs : 0;
            const int gw = (g >= p.band_lo && g <= p.band_hi) ? g : 0;   // rows with work here
            const long long items = ((static_cast<long long>(gw) + chunk - 1) / chunk) * item_tiles;
            nt_max = max(nt_max, gw >= chunk ? chunk : (gw + (kPair ? 31 : 15)) & (kPair ? ~31 : ~15));
            long long incl_r = g, incl_i = items;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const long long a = __shfl_up_sync(0xffffffffu, incl_r, d);
                const long long b = __shfl_up_sync(0xffffffffu, incl_i, d);
                if (lane >= d) {
                    incl_r += a;
                    incl_i += b;
                }
            }
            const long long end_r = run_rows + incl_r, end_i = run_items + incl_i;
            if (e < E) {
                if (end_r > p.rows || end_i > INT32_MAX) *bad_flag = 1;
                roff[e] = static_cast<int>(end_r - g);
                ioff[e] = static_cast<int>(end_i - items);
            }
            run_rows += __shfl_sync(0xffffffffu, incl_r, 31);
            run_items += __shfl_sync(0xffffffffu, incl_i, 31);
        }
        nt_max = __reduce_max_sync(0xffffffffu, nt_max);
        if (lane == 0) {
            if (run_rows != p.rows || run_items > INT32_MAX) *bad_flag = 1;
            roff[E] = static_cast<int>(run_rows);
            ioff[E] = static_cast<int>(run_items);
            *nt_max_slot = nt_max;
            *chunk_slot = chunk;
        }
    }
    __syncthreads();
    if (*bad_flag) {
        if (blockIdx.x == 0 && tid == 0) set_status(p.status, MOE_ERR_DATA);
        return;
    }
    const int total_items = ioff[E];
    if (cta >= total_items) return;                 // the same for both CTAs of a pair
    const int my_items = (total_items - cta + n_cta - 1) / n_cta;
    const int chunk = *chunk_slot;
    const int tile_cols = p.swiglu ? kBN / 2 : kBN;
    // Work item i of this CTA.  Pair: the pair tile covers two column tiles;
    // this CTA's is the one of its rank, and nt is a multiple of 32 so that
    // each CTA's half of the token rows is a multiple of 16.
    auto make_item = [&](int i) -> Item {
        Item it = decode_item(cta + i * n_cta, roff, ioff, E, item_tiles, chunk,
                              kPair ? 2 * tile_cols : tile_cols);
        if constexpr (kPair) {
            it.n0 += static_cast<int>(rank) * tile_cols;
            it.nt = (it.nvalid + 31) & ~31;
        }
        return it;
    };
    // The CTA's first kItemCache work items, decoded once (visible after the
    // barrier set-up's __syncthreads below); later ones are decoded on demand.
    for (int t = tid; t < my_items && t < kItemCache; t += kThreads) {
        const Item it = make_item(t);
        item_cache[t] = make_int4(it.e, it.row0, it.n0, it.nvalid | (it.nt << 16));
    }
    uint32_t *nv_tab = reinterpret_cast<uint32_t *>(smem + kOffNvTab);
    if constexpr (kNv) {
        for (int t = tid; t < 256; t += kThreads) nv_tab[t] = e4m3_scaled_pair(static_cast<uint32_t>(t));
    }
    auto get_item = [&](int i) -> Item {
        if (i >= kItemCache) return make_item(i);
        const int4 v = item_cache[i];
        Item it;
        it.e = v.x;
        it.row0 = v.y;
        it.n0 = v.z;
        it.nvalid = v.w & 0xFFFF;
        it.nt = v.w >> 16;
        return it;
    };
    const int KT = p.k_stages;                  // multiple of 4
    // Split mode: every band <= 32 rows.  Four issuers, one per converter
    // warpgroup, each accumulating its warpgroup's stages into its own
    // K-partial.  The activation tile of a code stage (the band's rows x 256 k,
    // four 64-k boxes) travels in the same ring slot as the codes, so it is
    // fetched as far ahead as the codes; a slot is free again once the 16
    // converter warps have read the codes and the 4 issuers' MMAs are done.
    // Single mode (wider bands): the code ring holds codes only and the
    // activations use eight 64-k slots of their own, released with the A
    // slot of the same stage.  Wide mode (a band over 128 rows, K8
    // activations): items of up to 256 tokens; one 256-column accumulator (the
    // epilogue of an item runs before the next item's first MMA), and five
    // 32 KB activation slots with their own ring, released by their own MMA
    // commits, because eight would not fit in shared memory.
    const int nt_max = *nt_max_slot;
    // The band class of the launch fixes the mode: nt_max <= 32 exactly when
    // band_hi <= 32.
    constexpr bool split = kSplit;
    const bool wide = !kSplit && chunk == kWideNT;
    // One 64-k activation tile: split mode nt_max rows (16-row boxes); single
    // and wide mode nt_max rounded up to 64 rows (64- and 32-row boxes, up to
    // four copies a stage); pair mode this CTA's half, nt_max / 2 rounded up to
    // 64 rows, so twice the slots fit.
    const uint32_t act_stage_bytes =
        kPair ? static_cast<uint32_t>(((nt_max / 2) + 63) & ~63) * 128u
              : static_cast<uint32_t>(nt_max <= kPartCols ? nt_max : (nt_max + 63) & ~63) * 128u;
    const uint32_t n_act = kPair ? kPairActSlots : (wide ? kWideActSlots : kSlots);
    // Ring slot: codes (16 KB), [split: activation tile], [scale tile, loaded
    // with every even code stage for itself and the next one].
    const uint32_t scale_off = kCodeStageBytes + (split ? 4u * act_stage_bytes : 0u);
    const uint32_t ring_stage_bytes = scale_off + (p.scale_tma ? kScaleTileBytes : 0u);
    // The ring depth is even: the converter pairs take alternate code stages,
    // so with an even depth each pair owns every other slot and the slot it
    // waits on was last consumed by the pair itself.  With an odd depth the
    // slot of stage c + 2 last held stage c - 1 of the other pair, whose copy
    // may still be in flight; the barrier would then be two phases behind and
    // its parity would read as complete.
    const uint32_t CS = min(static_cast<uint32_t>(kCodeStagesMax),
                            (kRingBytes - (split ? 0u : n_act * act_stage_bytes)) / ring_stage_bytes) &
                        ~1u;
    const uint32_t act_off = CS * ring_stage_bytes;     // single/wide mode: activation slots
    // TMEM columns: the accumulator buffers (two; one in wide mode), then the
    // eight A slots (two sets of four, one set per code-stage parity).  With
    // every band <= 16 rows the K-partials need only 16 columns each.
    const bool narrow = split && nt_max <= 16;
    const uint32_t per_wg = 2u;                            // A-slot sets in flight
    const uint32_t part_cols = narrow ? kPartCols / 2 : kPartCols;
    const uint32_t nbuf = wide ? 1u : 2u;                  // accumulator buffers
    const uint32_t acc_cols =
        split ? kIssuerWarps * part_cols : (wide ? static_cast<uint32_t>(kWideNT) : kAccCols);
    const uint32_t acol0 = nbuf * acc_cols;
    // Activation-slot barriers the act producer waits on: the A-slot pair
    // barriers in single mode (activation slot s is released with A slot s),
    // their own in wide mode.
    uint64_t *act_free = wide ? act_empty : slot_empty;
    // Issuers splitting the token columns of an item (single and wide mode).
    const int n_iss = wide ? kWideIssuers : kSingleIssuers;

    if (warp == 0) {
        if constexpr (kPair) tmem_alloc_pair(tmem_slot, kTmemCols);   // both CTAs, same address
        else tmem_alloc(tmem_slot, kTmemCols);
    }
    // Pair: the even CTA's a_full, act_full and acc_empty also count the odd
    // CTA's arrivals (its converter warps, its activation relay, its epilogue
    // warps); the pair commits arrive on both CTAs' slot_empty, act_empty and
    // acc_full.
    const uint32_t peer_arrivals = (kPair && rank == 0) ? 1u : 0u;
    if (tid == 0) {
        for (uint32_t i = 0; i < CS; ++i) {
            mbar_init(&code_full[i], 1);
            mbar_init(&code_empty[i], 4 * kConvWG / 2 + (split ? kIssuerWarps : 0));
        }
        for (int i = 0; i < kSlotsMax; ++i) {
            mbar_init(&a_full[i], 4 * (1 + peer_arrivals));
            mbar_init(&act_full[i], 1 + peer_arrivals);
            mbar_init(&slot_empty[i], split ? 1 : n_iss);
            mbar_init(&act_empty[i], n_iss);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], split ? kIssuerWarps : n_iss);
            mbar_init(&acc_empty[i], 4 * kConvWG * (1 + peer_arrivals));
        }
        for (int i = 0; i < kIssuerWarps; ++i) mbar_init(&final_bar[i], 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync();   // the peer's barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t code_smem = smem_u32(smem + kOffCode);
    const uint32_t act_smem = smem_u32(smem + act_off);
    const uint64_t lim = p.wait_limit_ns;

    if (warp < kIssuerWarps) {
        // ----------------------------------------------------------- MMA issuers
        // Split mode: issuer w issues the stages of converter warpgroup w
        // (every 4th stage) into K-partial w.  Single mode: issuers 0 and 1 issue
        // every stage, each for its own part of the item's token columns (the
        // first a multiple of 16, about half), into one accumulator.  Wide mode:
        // issuer 0 alone, all of the item's columns.  The whole warp runs the
        // loop (its values stay warp-uniform); one elected lane issues the MMAs
        // and the commits, always the same lane, so each commit covers its MMAs.
        const int w = warp;
        if (kPair && rank == 1 && w == 0) {
            // Pair, odd CTA: relay of its activation halves.  Once its own half
            // of a stage has landed, arrive on the even CTA's barrier of that
            // stage (which the issuer there waits on), in the producer's order.
            const uint32_t peer_act_full = cluster_addr(act_full, 0);
            Ring r;
            bool ok = true;
            for (int i = 0; i < my_items && ok; ++i)
                for (int ks = 0; ks < KT && ok; ++ks, r.next(n_act)) {
                    ok = warp_wait_bounded(&act_full[r.slot], r.phase, abort_flag, p.status, lim);
                    if (ok && lane == 0) mbar_arrive_cluster(peer_act_full + 8u * r.slot);
                    __syncwarp();
                }
        } else if (kPair ? (rank == 0 && w == 0) : (split || w < n_iss)) {
            Item it = get_item(0);
            // This issuer's token columns [c0, c0 + cn) of the item (single mode).
            auto my_cols = [&](int nt, uint32_t &c0, uint32_t &cn) {
                if (split || n_iss == 1) {
                    c0 = 0;
                    cn = nt;
                    return;
                }
                const uint32_t half = ((nt / 2) + 15) & ~15;
                c0 = w == 0 ? 0u : half;
                cn = w == 0 ? half : nt - half;
            };
            uint32_t c0, cn;
            my_cols(it.nt, c0, cn);
            constexpr uint32_t kM = kPair ? 256u : 128u;      // pair: both CTAs' 128 weight rows
            uint32_t idesc = idesc_bf16_f32(kM, cn ? cn : 16);
            Ring ring;                        // split mode: code stage of this issuer's stage
            const uint32_t d_part = split ? w * part_cols : 0;
            Ring sr;                          // this issuer's A-slot sequence
            bool ok = true;
            // Single mode: stages come in groups of four (KT is a multiple of 4), and
            // the eight barriers of a group are probed together, so the probe
            // latency is paid once per group; the MMAs of the four stages follow,
            // each stage's slot released by its own commit.  Wide mode: groups of
            // two (each stage is twice the MMA work, and only five activation
            // slots exist, so a group of four would wait for most of them); the
            // activation slots have their own ring and their own release commit.
            constexpr int kGroupMax = 4;
            const int grp = wide ? 2 : kGroupMax;
            Ring ar;                          // wide mode: activation-slot ring
            for (int i = 0; i < my_items && ok && !split; ++i) {
                const uint32_t buf = wide ? 0u : static_cast<uint32_t>(i & 1);
                const uint32_t acc_par = (wide ? static_cast<uint32_t>(i) : static_cast<uint32_t>(i >> 1)) & 1u;
                for (int kp = 0; kp < KT; kp += grp) {
                    if (kp == 0 && !warp_wait_bounded(&acc_empty[buf], acc_par ^ 1u, abort_flag,
                                                      p.status, lim)) {
                        ok = false;
                        break;
                    }
                    uint32_t sl[kGroupMax], ph[kGroupMax], al[kGroupMax], aph[kGroupMax];
                    bool ready = true;
#pragma unroll
                    for (int h = 0; h < kGroupMax; ++h) {
                        if (h >= grp) break;
                        sl[h] = sr.slot;
                        ph[h] = sr.phase;
                        sr.next(kSlots);
                        if (wide) {
                            al[h] = ar.slot;
                            aph[h] = ar.phase;
                            ar.next(n_act);
                        } else {
                            al[h] = sl[h];
                            aph[h] = ph[h];
                        }
                        // A slots come in pairs (slot 2w, 2w + 1 of warpgroup w), and a
                        // group starts at an even slot: one barrier per pair.
                        if ((h & 1) == 0) ready = ready & mbar_try_wait(&a_full[sl[h] >> 1], ph[h]);
                        ready = ready & mbar_try_wait(&act_full[al[h]], aph[h]);
                    }
                    if (!__all_sync(0xffffffffu, ready)) {
#pragma unroll
                        for (int h = 0; h < kGroupMax; ++h)
                            if (h < grp && ok &&
                                (((h & 1) == 0 &&
                                  !warp_wait_bounded(&a_full[sl[h] >> 1], ph[h], abort_flag, p.status, lim)) ||
                                 !warp_wait_bounded(&act_full[al[h]], aph[h], abort_flag, p.status,
                                                    lim)))
                                ok = false;
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * acc_cols + c0;
                    if (elect_one()) {
#pragma unroll
                        for (int h = 0; h < kGroupMax; ++h) {
                            if (h >= grp) break;
                            const uint32_t a_col = tmem_base + acol0 + sl[h] * kAColsPerSlot;
                            const uint64_t b0 =
                                smem_desc_sw128(act_smem + al[h] * act_stage_bytes + c0 * 128);
                            if (cn > 0)
#pragma unroll
                            for (int kk = 0; kk < kStageK / 16; ++kk)
                                mma_issue(d_tmem, a_col + kk * 8,
                                            b0 + static_cast<uint64_t>(kk * 2), idesc,
                                            (kp == 0 && h == 0 && kk == 0) ? 0u : 1u);
                            if (h & 1) mma_commit_all(&slot_empty[sl[h] >> 1]);
                            if (wide) mma_commit_all(&act_empty[al[h]]);
                        }
                        if (kp + grp >= KT) mma_commit_all(&acc_full[buf]);
                    }
                    __syncwarp();
                }
                if (ok && i + 1 < my_items) {
                    it = get_item(i + 1);
                    my_cols(it.nt, c0, cn);
                    idesc = idesc_bf16_f32(kM, cn ? cn : 16);
                }
            }
            // Split mode: issuer w issues sub-stages 2w and 2w + 1 of every code
            // stage (8 MMAs, in k order) into its K-partial w.
            for (int i = 0; i < my_items && ok && split; ++i) {
                const uint32_t buf = i & 1;
                for (int m = 0; m < KT / 4; ++m) {
                    if (m == 0 && !warp_wait_bounded(&acc_empty[buf], ((i >> 1) & 1) ^ 1,
                                                     abort_flag, p.status, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t s0 = 2u * w + 4u * sr.slot, par = sr.phase;   // sub-stage 2w at slot set
                    // One probe for both barriers (the usual case: both complete).
                    const bool ready = __all_sync(
                        0xffffffffu, mbar_try_wait(&a_full[s0 >> 1], par) &
                                         mbar_try_wait(&code_full[ring.slot], ring.phase));
                    if (!ready &&
                        (!warp_wait_bounded(&a_full[s0 >> 1], par, abort_flag, p.status, lim) ||
                         !warp_wait_bounded(&code_full[ring.slot], ring.phase, abort_flag,
                                            p.status, lim))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * acc_cols + d_part;
                    const uint32_t b_base = code_smem + ring.slot * ring_stage_bytes +
                                            kCodeStageBytes + 2u * w * act_stage_bytes;
                    if (elect_one()) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t a_col = tmem_base + acol0 + (s0 + h) * kAColsPerSlot;
                            const uint64_t b0 = smem_desc_sw128(b_base + h * act_stage_bytes);
#pragma unroll
                            for (int kk = 0; kk < kStageK / 16; ++kk)
                                mma_issue(d_tmem, a_col + kk * 8,
                                            b0 + static_cast<uint64_t>(kk * 2), idesc,
                                            (m == 0 && h == 0 && kk == 0) ? 0u : 1u);
                        }
                        mma_commit_all(&slot_empty[s0 >> 1]);
                        mma_commit_all(&code_empty[ring.slot]);
                        if (m + 1 == KT / 4) mma_commit_all(&acc_full[buf]);
                    }
                    __syncwarp();
                    ring.next(CS);
                    sr.next(per_wg);
                }
                if (ok && i + 1 < my_items) {
                    it = get_item(i + 1);
                    my_cols(it.nt, c0, cn);
                    idesc = idesc_bf16_f32(128, cn ? cn : 16);
                }
            }
            // All MMAs issued by the elected lane must finish before TMEM is freed.
            if (elect_one()) mma_commit_own(&final_bar[w]);
            __syncwarp();
            warp_wait_bounded(&final_bar[w], 0, nullptr, p.status, lim);
        }
    } else if (warp == kCodeWarp) {
        // ------------------------------------------------------ code producer
        // Converged warp, one elected lane issues the copies.  Split mode: the
        // band's activation tile of the code stage rides along; with bands of
        // <= 16 rows and K % 256 == 0 it is one 3-D box (16 rows x 4 x 64 k,
        // stored as four 64-k tiles), else 2-D boxes of 16 rows x 64 k.
        const bool use3d = p.act3d && narrow;    // one 16-row group per code stage
        constexpr bool gather = kMap == kMapGather;
        if (lane == 0) {
            tma_prefetch_map(&tm_codes);
            if (split) tma_prefetch_map(use3d ? &tm_act3 : &tm_act);
            if (p.scale_tma) tma_prefetch_map(&tm_scales);
        }
        // Fused SwiGLU: tile rows 32q .. 32q + 15 are gate rows n0 + 16q .. +15
        // and 32q + 16 .. 32q + 31 the matching up rows (I further on).  The
        // maps tm_codes / tm_scales then view each expert's rows as
        // [16-row group q][half][row i] (5-D, x innermost), so one box of
        // {x, 16 rows, 2 halves, 4 groups, 1 expert} lands the whole tile in
        // that order; groups past I/16 are zero-filled.
        __syncwarp();
        Ring r;
        uint32_t issued = 0;
        bool ok = true;
        for (int i = 0; i < my_items && ok; ++i) {
            const Item it = get_item(i);
            const int y = it.e * p.N + it.n0;
            // Gather (split mode, nt <= 32): lane l holds the activation row of
            // the item's row l; rows past the band repeat its first row (their
            // outputs are never written).
            int act_row = 0;
            if constexpr (split && gather)
                act_row = gather_row(p, it.row0 + (lane < it.nvalid ? lane : 0));
            for (int kc = 0; kc < KT / 4; ++kc, r.next(CS), ++issued) {
                if (!warp_wait_bounded(&code_empty[r.slot], r.phase ^ 1u, abort_flag, p.status,
                                       lim)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    const uint32_t dst = code_smem + r.slot * ring_stage_bytes;
                    const bool scales_here = p.scale_tma != 0;
                    mbar_arrive_expect_tx(&code_full[r.slot],
                                          kCodeStageBytes + (split ? it.nt * 512u : 0u) +
                                              (scales_here ? kScaleTileBytes : 0u));
                    // 16 bytes a row: MXFP4 this code stage and its even/odd twin;
                    // NVFP4 this code stage's sixteen per-16 scales.
                    const int sx = kNv ? kc * 16 : (kc & ~1) * 8;
                    if (p.swiglu) {
                        tma_load_5d(dst, &tm_codes, kc * 128, 0, 0, it.n0 >> 4, it.e,
                                    &code_full[r.slot]);
                        if (scales_here)
                            tma_load_5d(dst + scale_off, &tm_scales, sx, 0, 0, it.n0 >> 4, it.e,
                                        &code_full[r.slot]);
                    } else {
                        tma_load_2d(dst, &tm_codes, kc * 128, y, &code_full[r.slot]);
                        if (scales_here)
                            tma_load_2d(dst + scale_off, &tm_scales, sx, y, &code_full[r.slot]);
                    }
                    if (split && !gather) {
                        for (int grp = 0; grp < it.nt / 16; ++grp) {
                            if (use3d) {
                                tma_load_3d(dst + kCodeStageBytes + grp * 2048, &tm_act3, 0,
                                            it.row0 + grp * 16, kc * 4, &code_full[r.slot]);
                            } else {
                                for (int sub = 0; sub < 4; ++sub)
                                    tma_load_2d(dst + kCodeStageBytes + sub * act_stage_bytes +
                                                    grp * 2048,
                                                &tm_act, kc * kCodeK + sub * kStageK,
                                                it.row0 + grp * 16, &code_full[r.slot]);
                            }
                        }
                    }
                }
                __syncwarp();
                if constexpr (split && gather) {
                    // Lane l < nt / 4 gathers rows 4l .. 4l + 3 of the four 64-k
                    // sub-stages (after the elected lane's expect_tx above).
                    const int q = 4 * (lane & 7);
                    const int r0 = __shfl_sync(0xffffffffu, act_row, q);
                    const int r1 = __shfl_sync(0xffffffffu, act_row, q + 1);
                    const int r2 = __shfl_sync(0xffffffffu, act_row, q + 2);
                    const int r3 = __shfl_sync(0xffffffffu, act_row, q + 3);
                    if (lane < it.nt / 4) {
                        const uint32_t dst = code_smem + r.slot * ring_stage_bytes + kCodeStageBytes +
                                             static_cast<uint32_t>(lane) * 512u;
                        for (int sub = 0; sub < 4; ++sub)
                            tma_gather4(dst + sub * act_stage_bytes, &tm_act, kc * kCodeK + sub * kStageK,
                                        r0, r1, r2, r3, &code_full[r.slot]);
                    }
                    __syncwarp();
                }
            }
        }
        if (!ok && lane == 0) {   // drain: every issued copy must land before the CTA exits
            const uint32_t first = issued > CS ? issued - CS : 0;
            for (uint32_t h = first; h < issued; ++h)
                wait_bounded(&code_full[h % CS], (h / CS) & 1u, nullptr, p.status, lim);
        }
    } else if (warp == kActWarp && kMap == kMapGather) {
        // ------------------- activation producer with the gather (single, wide)
        // Lane 0 waits for the slot and posts the byte count; lane l then gathers
        // rows 8l .. 8l + 7 of the item with two four-row TMA gathers.
        if (!split) {
            if (lane == 0) tma_prefetch_map(&tm_act64);
            Ring r;
            uint32_t issued = 0;
            bool ok = true;
            for (int i = 0; i < my_items && ok; ++i) {
                const Item it = get_item(i);
                int ar[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // activation rows of rows 8l .. 8l + 7
                if (8 * lane < it.nt) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int rr = 8 * lane + q;   // rows past the band repeat its first row
                        ar[q] = gather_row(p, it.row0 + (rr < it.nvalid ? rr : 0));
                    }
                }
                for (int ks = 0; ks < KT; ++ks, r.next(n_act), ++issued) {
                    int free_ok = 1;
                    if (lane == 0) {
                        free_ok = wait_bounded(wide ? &act_free[r.slot] : &act_free[r.slot >> 1],
                                               r.phase ^ 1u, abort_flag, p.status, lim);
                        if (free_ok)
                            mbar_arrive_expect_tx(&act_full[r.slot], static_cast<uint32_t>(it.nt) * 128u);
                    }
                    if (!__shfl_sync(0xffffffffu, free_ok, 0)) {
                        ok = false;
                        break;
                    }
                    if (8 * lane < it.nt) {   // nt is a multiple of 16: all eight rows exist
                        const uint32_t d = act_smem + r.slot * act_stage_bytes +
                                           static_cast<uint32_t>(lane) * 1024u;
                        tma_gather4(d, &tm_act64, ks * kStageK, ar[0], ar[1], ar[2], ar[3],
                                    &act_full[r.slot]);
                        tma_gather4(d + 512u, &tm_act64, ks * kStageK, ar[4], ar[5], ar[6], ar[7],
                                    &act_full[r.slot]);
                    }
                }
            }
            if (!ok && lane == 0) {   // drain: every issued copy must land before the CTA exits
                const uint32_t first = issued > n_act ? issued - n_act : 0;
                for (uint32_t h = first; h < issued; ++h)
                    wait_bounded(&act_full[h % n_act], (h / n_act) & 1u, nullptr, p.status, lim);
            }
        }
    } else if (warp == kActWarp) {
        // ------------------------------------- activation producer (single mode)
        if (lane == 0 && !split) {
            tma_prefetch_map(&tm_act64);
            tma_prefetch_map(&tm_act3);
            Ring r;
            uint32_t issued = 0;
            bool ok = true;
            for (int i = 0; i < my_items && ok; ++i) {
                const Item it = get_item(i);
                for (int ks = 0; ks < KT; ++ks, r.next(n_act), ++issued) {
                    // Single mode: activation slot s is free with A slot s, whose
                    // barrier is shared with the other slot of its pair.
                    if (!wait_bounded(wide ? &act_free[r.slot] : &act_free[r.slot >> 1], r.phase ^ 1u,
                                      abort_flag, p.status, lim)) {
                        ok = false;
                        break;
                    }
                    // The stage's token rows (pair: this CTA's half of them) in 64-row
                    // boxes.  Pair: a last part of at most 32 rows takes a 32-row box
                    // (tm_act3 holds the 32-row map in these launches); copies cost
                    // the SM per request as well as per byte, so smaller boxes would
                    // lose more than the at most 16 rows they save.  One CTA: whole
                    // 64-row boxes (measured faster there).
                    const uint32_t dst = act_smem + r.slot * act_stage_bytes;
                    const int n = kPair ? it.nt / 2 : it.nt;
                    const int r0 = it.row0 + static_cast<int>(rank) * n;
                    const int full64 = n & ~63, tail = n - full64;
                    const int fetched =
                        full64 + (tail == 0 ? 0 : ((kPair && tail <= 32) ? 32 : 64));
                    mbar_arrive_expect_tx(&act_full[r.slot], static_cast<uint32_t>(fetched) * 128u);
                    for (int g = 0; g < full64; g += 64)
                        tma_load_2d(dst + g * 128, &tm_act64, ks * kStageK, r0 + g, &act_full[r.slot]);
                    if (tail > 32 || (!kPair && tail > 0))
                        tma_load_2d(dst + full64 * 128, &tm_act64, ks * kStageK, r0 + full64,
                                    &act_full[r.slot]);
                    else if (tail > 0)
                        tma_load_2d(dst + full64 * 128, &tm_act3, ks * kStageK, r0 + full64,
                                    &act_full[r.slot]);
                }
            }
            if (!ok) {
                const uint32_t first = issued > n_act ? issued - n_act : 0;
                for (uint32_t h = first; h < issued; ++h)
                    wait_bounded(&act_full[h % n_act], (h / n_act) & 1u, nullptr, p.status, lim);
            }
        }
    } else {
        // ------------------------------------------------ converters + epilogue
        // The warpgroups work in pairs on alternate code stages: warpgroups 0 and
        // 1 on the even ones, 2 and 3 on the odd ones, each taking one 128-k half
        // (sub-stages 2h and 2h + 1).  A thread reads the 64 code bytes of its
        // weight row (TMEM lane) in the half, decodes them into 64 bf16 pairs
        // (K8-interleaved reduction order) and stores them, 32 columns at a
        // time, into the warpgroup's two A slots 2wg and 2wg + 1; the slots are
        // reused every other code stage of the warpgroup.  Every warpgroup also
        // writes its quarter of the token columns of item i - 2 once it has gone
        // past item i - 1, and of the remaining items at the end.
        const int wg = (warp - kConvWarp0) >> 2;
        const int pair = wg >> 1;                  // code-stage parity of this warpgroup
        const int half = wg & 1;                   // which 128-k half of the code stage
        const int wtid = tid - 32 * kConvWarp0 - 128 * wg;   // 0..127 within the warpgroup
        const int q = warp & 3;                    // TMEM lane quarter = warp within the group
        const int row = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t slot0 = 2u * wg;            // A slots 2wg, 2wg + 1
        const uint32_t a_base = tmem_base + lane_off + acol0 + slot0 * kAColsPerSlot;
        const int KT4 = KT / 4;
        // This row's four swizzled 16-byte chunks of the half.
        uint32_t chunk_off[4];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
            chunk_off[ch] = row * 128 + (((4 * half + ch) ^ (row & 7)) << 4);
        int bad_scale = 0;
        bool ok = true;
        // Weight row of this thread's tile row in item `it` (fused SwiGLU: the
        // gate/up interleave of the tile).
        auto weight_row = [&](const Item &it) -> int {
            return p.swiglu ? it.n0 + swiglu_row_offset(row) + (swiglu_row_is_up(row) ? p.I : 0)
                            : it.n0 + row;
        };
        // Scale bytes of code stage m for this row and half: 32-k blocks 8m + 4h
        // .. 8m + 4h + 3 of the row, each reading scale byte blk >> scale_shift
        // (one byte per 32 k, or per 512 k).  A tile row beyond N reads row N - 1
        // (its codes are zero-filled, so the value never matters).
        auto scale_base = [&](int j) -> const uint8_t * {
            const Item it = get_item(j);
            const int n = min(weight_row(it), p.N - 1);
            return p.scales + (static_cast<size_t>(it.e) * p.N + n) * p.scale_row +
                   (kNv ? 8 * half : 0);
        };
        auto load_scales = [&](const uint8_t *sb, int m) -> uint32_t {
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int blk = 8 * m + 4 * half + b;
                const uint32_t sbyte =
                    blk < p.k_blocks ? static_cast<uint32_t>(__ldg(sb + (blk >> p.scale_shift))) : 127u;
                v |= sbyte << (8 * b);
            }
            return v;
        };
        // NVFP4: the eight per-16 scale bytes of code stage m for this row and
        // half (blocks 16m + 8h .. 16m + 8h + 7); blocks past K read 1.0 (0x38).
        auto load_scales_nv = [&](const uint8_t *sbase, int m) -> uint2 {
            uint32_t v[2] = {0u, 0u};
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int blk = 16 * m + 8 * half + b;
                const uint32_t sbyte =
                    blk < p.scale_row ? static_cast<uint32_t>(__ldg(sbase + 16 * m + b)) : 0x38u;
                v[b >> 2] |= sbyte << (8 * (b & 3));
            }
            return make_uint2(v[0], v[1]);
        };
        auto epilogue = [&](int i) -> bool {
            const uint32_t buf = wide ? 0u : static_cast<uint32_t>(i & 1);
            const uint32_t par = (wide ? static_cast<uint32_t>(i) : static_cast<uint32_t>(i >> 1)) & 1u;
            if (!warp_wait_bounded(&acc_full[buf], par, abort_flag, p.status, lim))
                return false;
            tc_fence_after();
            const Item it = get_item(i);
            const float ts = kNv ? __ldg(ws2 + it.e) : 0.0f;
            if (wide)
                store_item_wide<kNv, kMap == kMapScatter>(p, it, tmem_base + lane_off, wg, row, ts);
            else
                store_item<kNv, kMap == kMapScatter>(p, it, tmem_base + lane_off + buf * acc_cols, wg, row, split,
                                part_cols, ts);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (kPair && rank == 1) mbar_arrive_cluster(cluster_addr(&acc_empty[buf], 0));
                else mbar_arrive(&acc_empty[buf]);
            }
            return true;
        };
        const uint32_t total_cs = static_cast<uint32_t>(my_items) * KT4;
        Ring code;                                 // ring position of code stage c
        if (pair) code.next(CS);
        uint32_t sphase = 0;                       // A-slot phase: (c / 2) & 1
        int i = pair / KT4, m = pair % KT4;        // item and code stage within it
        int ep_next = 0;                           // next item whose output this warp writes
        int cur_nt = 0;
        bool row_ok = false;
        const uint8_t *sb = nullptr;
        auto enter_item = [&](int it_idx) {
            const Item it = get_item(it_idx);
            cur_nt = it.nt;
            // Scale bytes of a tile row beyond N (read with the tile) never count
            // as errors: those rows are not part of the output.
            row_ok = p.swiglu ? it.n0 + swiglu_row_offset(row) < p.I : it.n0 + row < p.N;
            if (!p.scale_tma) sb = scale_base(it_idx);
        };
        if (i < my_items) enter_item(i);
        // Barrier tests are issued ahead of their use (non-blocking), so their
        // latency hides behind the decode: the next code stage's at the start of
        // this stage's decode, this stage's A slots just before it.  A test that
        // fails falls back to the bounded wait.
        bool code_ready = false;
        for (uint32_t c = pair; c < total_cs && ok; c += 2) {
            if (!__all_sync(0xffffffffu, code_ready) &&
                !warp_wait_bounded(&code_full[code.slot], code.phase, abort_flag, p.status,
                                   lim)) {
                ok = false;
                break;
            }
            uint8_t *slot_base = smem + kOffCode + code.slot * ring_stage_bytes;
            const uint32_t sw =
                kNv ? 0u
                    : (p.scale_tma ? *reinterpret_cast<const uint32_t *>(slot_base + scale_off +
                                                                         row * 16 + (m & 1) * 8 +
                                                                         4 * half)
                                   : load_scales(sb, m));
            uint2 swn = make_uint2(0u, 0u);        // NVFP4: sub-stage h's four per-16 scales
            if constexpr (kNv) {
                swn = p.scale_tma ? *reinterpret_cast<const uint2 *>(slot_base + scale_off +
                                                                     row * 16 + 8 * half)
                                  : load_scales_nv(sb, m);
                // E4M3 NaN bytes (low seven bits all set) are errors.
                const uint32_t nan = (((swn.x & 0x7F7F7F7Fu) + 0x01010101u) |
                                      ((swn.y & 0x7F7F7F7Fu) + 0x01010101u)) & 0x80808080u;
                if (nan && row_ok) bad_scale = 1;
            }
            uint32_t cw[4][4];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const uint4 v = *reinterpret_cast<const uint4 *>(slot_base + chunk_off[ch]);
                cw[ch][0] = v.x;
                cw[ch][1] = v.y;
                cw[ch][2] = v.z;
                cw[ch][3] = v.w;
            }
            // The ring slot is refilled by TMA (the async proxy) once released:
            // order these generic-proxy reads of it before that write.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&code_empty[code.slot]);
            if (!p.act_k8) {
                // Interleave every 16-byte chunk of the two sub-stages' activation
                // rows in place (the permutation stays inside a chunk, so the
                // swizzle of the tile does not matter).
                if (!split &&
                    (!warp_wait_bounded(&act_full[slot0], sphase, abort_flag, p.status, lim) ||
                     !warp_wait_bounded(&act_full[slot0 + 1], sphase, abort_flag, p.status,
                                        lim))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint4 *abase = reinterpret_cast<uint4 *>(
                        split ? slot_base + kCodeStageBytes + (2 * half + h) * act_stage_bytes
                              : smem + act_off + (slot0 + h) * act_stage_bytes);
                    for (int cc = wtid; cc < cur_nt * 8; cc += 128)
                        abase[cc] = interleave8(abase[cc]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            const bool slots_ready = mbar_test_wait(&slot_empty[wg], sphase ^ 1u);
            // Ring position of this pair's next code stage, c + 2 (one wrap at
            // most: the depth is at least 2).
            Ring nx = code;
            nx.slot += 2;
            if (nx.slot >= CS) {
                nx.slot -= CS;
                nx.phase ^= 1u;
            }
            code_ready = c + 2 < total_cs && mbar_test_wait(&code_full[nx.slot], nx.phase);
            // Scale bytes 0..128 take one bf16 FMA, 129..252 two, 253..255 are
            // errors; the warp agrees on the path.  A byte is above 128 exactly
            // when its top bit and one of its low seven bits are set.
            const uint32_t big = sw & ((sw & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) & 0x80808080u;
            const bool slow = !kNv && __any_sync(0xffffffffu, big != 0);
            if (!__all_sync(0xffffffffu, slots_ready) &&
                !warp_wait_bounded(&slot_empty[wg], sphase ^ 1u, abort_flag, p.status, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {          // sub-stage 2·half + h -> A slot slot0 + h
                uint32_t o[32];
                if constexpr (kNv) {
                    // Per-16 blocks: words 0-1 and 2-3 of each 32-code chunk.
                    const uint32_t sv = h ? swn.y : swn.x;
                    decode16_scaled(cw[2 * h][0], cw[2 * h][1], nv_tab[sv & 0xFFu], &o[0]);
                    decode16_scaled(cw[2 * h][2], cw[2 * h][3], nv_tab[(sv >> 8) & 0xFFu], &o[8]);
                    decode16_scaled(cw[2 * h + 1][0], cw[2 * h + 1][1], nv_tab[(sv >> 16) & 0xFFu],
                                    &o[16]);
                    decode16_scaled(cw[2 * h + 1][2], cw[2 * h + 1][3], nv_tab[sv >> 24], &o[24]);
                } else {
                if (__builtin_expect(!slow, 1)) {
                    // Scale byte b of sw in both 16-bit halves, then 2^(s-1) as bf16x2.
                    const uint32_t sp0 = prmt(sw, 0u, h ? 0x4242u : 0x4040u);
                    const uint32_t sp1 = prmt(sw, 0u, h ? 0x4343u : 0x4141u);
                    decode32_single(cw[2 * h], sp0 * 0x80u + 0x3F003F00u, &o[0]);
                    decode32_single(cw[2 * h + 1], sp1 * 0x80u + 0x3F003F00u, &o[16]);
                } else {
                    if (!decode32_any(cw[2 * h], (sw >> (16 * h)) & 0xFFu, &o[0]) && row_ok)
                        bad_scale = 1;
                    if (!decode32_any(cw[2 * h + 1], (sw >> (16 * h + 8)) & 0xFFu, &o[16]) && row_ok)
                        bad_scale = 1;
                }
                }
                __syncwarp();
                tmem_st32(a_base + h * kAColsPerSlot, o);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (kPair && rank == 1) mbar_arrive_cluster(cluster_addr(&a_full[wg], 0));
                else mbar_arrive(&a_full[wg]);
            }
            // Wide mode has one accumulator: the next item's first MMAs wait for
            // this item's epilogue.  The slots this pair fills next were last
            // read by its stage c, whose MMAs needed the epilogue of item i - 1,
            // so that epilogue runs now, right after the pair's first stage of
            // item i (its decode-ahead stays in flight meanwhile).
            if (wide) {
                while (ok && ep_next <= i - 1) {
                    if (!epilogue(ep_next)) ok = false;
                    ++ep_next;
                }
            }
            // Next code stage of this pair: c + 2.
            code = nx;
            sphase ^= 1u;
            m += 2;
            while (m >= KT4) {
                m -= KT4;
                ++i;
                while (ok && ep_next <= i - 2) {
                    if (!epilogue(ep_next)) ok = false;
                    ++ep_next;
                }
                if (i < my_items) enter_item(i);
            }
        }
        // Outputs of the items not written yet.
        while (ok && ep_next < my_items) {
            if (!epilogue(ep_next)) ok = false;
            ++ep_next;
        }
        if (bad_scale) set_status(p.status, MOE_ERR_DATA);
    }

    // ---------------------------------------------------------------- teardown
    // Pair: neither CTA frees its tensor memory or leaves while the pair's MMAs,
    // commits or the peer's arrivals may still reach it.
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync();
    tc_fence_after();
    if (warp == 0) {
        __syncwarp();
        if constexpr (kPair) tmem_dealloc_pair(tmem_base, kTmemCols);
        else tmem_dealloc(tmem_base, kTmemCols);
    }
    if constexpr (kPair) cluster_sync();
}

template <bool kSplit, int kMap>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_codes,
                    const __grid_constant__ CUtensorMap tm_act,
                    const __grid_constant__ CUtensorMap tm_act3,
                    const __grid_constant__ CUtensorMap tm_scales,
                    const __grid_constant__ CUtensorMap tm_act64, const Params p) {
    gemm_body<false, kSplit, kMap>(tm_codes, tm_act, tm_act3, tm_scales, tm_act64, p, nullptr);
}

// Wide bands in CTA pairs (clusters of two): M = 256 MMAs over two SMs.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_codes,
                         const __grid_constant__ CUtensorMap tm_act,
                         const __grid_constant__ CUtensorMap tm_act3,
                         const __grid_constant__ CUtensorMap tm_scales,
                         const __grid_constant__ CUtensorMap tm_act64, const Params p) {
    gemm_body<false, false, kMapNone, true>(tm_codes, tm_act, tm_act3, tm_scales, tm_act64, p,
                                            nullptr);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
grouped_gemm_nvfp4_pair_kernel(const __grid_constant__ CUtensorMap tm_codes,
                               const __grid_constant__ CUtensorMap tm_act,
                               const __grid_constant__ CUtensorMap tm_act3,
                               const __grid_constant__ CUtensorMap tm_scales,
                               const __grid_constant__ CUtensorMap tm_act64, const Params p,
                               const float *__restrict__ ws2) {
    gemm_body<true, false, kMapNone, true>(tm_codes, tm_act, tm_act3, tm_scales, tm_act64, p, ws2);
}

template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_codes,
                          const __grid_constant__ CUtensorMap tm_act,
                          const __grid_constant__ CUtensorMap tm_act3,
                          const __grid_constant__ CUtensorMap tm_scales,
                          const __grid_constant__ CUtensorMap tm_act64, const Params p,
                          const float *__restrict__ ws2) {
    gemm_body<true, kSplit, kMapNone>(tm_codes, tm_act, tm_act3, tm_scales, tm_act64, p, ws2);
}

// Debug view of the decode: one thread per (weight row n, 32-element block); the
// GEMM's decode routine, with the reduction order mapped back to natural k.
__global__ void decode_expert_kernel(const uint8_t *codes, const uint8_t *scales, int N, int K,
                                     int e, uint16_t *out, int *status) {
    const int nblk = K / 32;
    const long long total = static_cast<long long>(N) * nblk;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(i / nblk), b = static_cast<int>(i % nblk);
        const size_t row = static_cast<size_t>(e) * N + n;
        const uint8_t *src = codes + row * (K / 2) + b * 16;
        uint32_t c[4];
        for (int w = 0; w < 4; ++w)
            c[w] = static_cast<uint32_t>(src[4 * w]) | (static_cast<uint32_t>(src[4 * w + 1]) << 8) |
                   (static_cast<uint32_t>(src[4 * w + 2]) << 16) |
                   (static_cast<uint32_t>(src[4 * w + 3]) << 24);
        const uint32_t s = scales[row * nblk + b];
        uint32_t o[16];
        if (s <= 128u) decode32_single(c, scale_pair_single(s), o);
        else if (!decode32_any(c, s, o)) set_status(status, MOE_ERR_DATA);
        uint4 *dst = reinterpret_cast<uint4 *>(out + static_cast<size_t>(n) * K + b * 32);
        for (int w = 0; w < 4; ++w)
            dst[w] = deinterleave8(make_uint4(o[4 * w], o[4 * w + 1], o[4 * w + 2], o[4 * w + 3]));
    }
}

// Failure-detection self-test: wait on a barrier that never completes.
__global__ void bounded_wait_kernel(uint64_t limit_ns, int *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) wait_bounded(&bar, 0, &abort_flag, status, limit_ns);
}

}  // namespace gemm

// ----------------------------------------------------------------- host side

// CTA-pair use for the launch of longer bands (process-wide): 0 automatic,
// 1 never, 2 whenever the shape allows it.
static std::atomic<int> g_pair_mode{0};

void set_gemm_pairing(int mode) { g_pair_mode.store(mode, std::memory_order_relaxed); }

// Clusters of two that the device can keep resident at once with the pair
// kernel's shared memory (looked up once per device and weight format).
template <bool kNv>
static int pair_clusters(int num_sms, int smem_bytes) {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cached[dev].load(std::memory_order_acquire);
    if (n == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
        cfg.blockDim = dim3(gemm::kThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
        int clusters = 0;
        const cudaError_t e =
            kNv ? cudaOccupancyMaxActiveClusters(&clusters, gemm::grouped_gemm_nvfp4_pair_kernel, &cfg)
                : cudaOccupancyMaxActiveClusters(&clusters, gemm::grouped_gemm_pair_kernel, &cfg);
        if (e != cudaSuccess)
            clusters = 0;
        n = clusters > 0 ? clusters : -1;
        cached[dev].store(n, std::memory_order_release);
    }
    return n > 0 ? n : 0;
}

// The driver's tensor-map encoder, looked up once per process (a function-local
// static is initialised once even when host threads race on the first call).
static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }();
    return fn;
}

// Both weight formats.  kNv = false: `scales` are per-32 E8M0 bytes [E, N, K/32].
// kNv = true: `scales` are per-16 E4M3 bytes [E, N, K/16] and ws2 the per-expert
// f32 weight_scale_2.
// swiglu: N = 2 * I weight rows ([gate | up]); `out` is h, bf16 [rows, I], in
// the K8-interleaved order when h_k8.
// scale_block (MXFP4): consecutive k per E8M0 scale byte, 32 or 512.
// kMap == kMapGather: sorted row r reads activation row gather_slot[r] /
// gather_k of act [act_rows, K] (K8-interleaved).  kMap == kMapScatter: sorted
// row r is written to output row out_row[r].
template <bool kNv, int kMap = gemm::kMapNone>
static moe_status launch_gemm(const uint16_t *act, int rows, int K, const uint8_t *codes,
                              const uint8_t *scales, const float *ws2, const int32_t *group_sizes,
                              int E, int N, void *out, int out_bf16, int act_k8, int swiglu,
                              int h_k8, int *status, uint64_t wait_limit_ns, cudaStream_t stream,
                              int num_sms, int scale_block = 32,
                              const int32_t *gather_slot = nullptr, int gather_k = 1,
                              int act_rows = 0, const int32_t *out_row = nullptr) {
    static_assert(!kNv || kMap == gemm::kMapNone, "row maps are built for MXFP4 only");
    using namespace gemm;
    if (rows == 0) return MOE_OK;
    const int I = N / 2;   // fused SwiGLU: gate rows [0, I), up rows [I, 2I); I % 16 == 0
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
    if (!encode) return MOE_ERR_CUDA;

    CUtensorMap tm_codes, tm_act, tm_act3, tm_scales, tm_act64;
    // Fused SwiGLU: the rows of a weight tensor with `row_bytes` bytes a row,
    // seen as [E][I/16 groups][2 halves][16 rows][row_bytes] with the group
    // and half dimensions swapped in the view, so one box holds the tile's
    // rows in the order (group, half, row).
    auto encode_swiglu_view = [&](CUtensorMap *map, const void *base, cuuint64_t row_bytes,
                                  cuuint32_t box_x, CUtensorMapSwizzle swz) -> bool {
        cuuint64_t dims[5] = {row_bytes, 16, 2, static_cast<cuuint64_t>(I / 16),
                              static_cast<cuuint64_t>(E)};
        cuuint64_t strides[4] = {row_bytes, static_cast<cuuint64_t>(I) * row_bytes, 16 * row_bytes,
                                 static_cast<cuuint64_t>(N) * row_bytes};
        cuuint32_t box[5] = {box_x, 16, 2, 4, 1};
        cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(base), dims, strides,
                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (swiglu) {
        if (!encode_swiglu_view(&tm_codes, codes, static_cast<cuuint64_t>(K / 2), 128,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return MOE_ERR_CUDA;
    } else {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2),
                              static_cast<cuuint64_t>(E) * static_cast<cuuint64_t>(N)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
        cuuint32_t box[2] = {128, 128};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return MOE_ERR_CUDA;
    }
    // Activation boxes of 64 k by 16 rows (split mode) and by 64 rows (single
    // and wide mode); with the gather both maps are one row high (gather4).
    constexpr bool gather = kMap == kMapGather;
    const cuuint64_t map_rows = static_cast<cuuint64_t>(gather ? act_rows : rows);
    {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), map_rows};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        cuuint32_t box[2] = {64, gather ? 1u : 16u};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(act), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return MOE_ERR_CUDA;
    }
    {   // 64-row boxes for wide bands
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), map_rows};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        cuuint32_t box[2] = {64, gather ? 1u : 64u};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_act64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(act), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return MOE_ERR_CUDA;
    }
    // 32-row boxes: the last part of a stage's rows in the launches for longer
    // bands (passed there in place of the split mode's 3-D map).
    CUtensorMap tm_act32;
    if (!gather) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), map_rows};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        cuuint32_t box[2] = {64, 32};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_act32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(act), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return MOE_ERR_CUDA;
    } else {
        tm_act32 = tm_act;
    }
    // The same activations seen as [K/64 chunks][rows][64]: one box holds 16
    // rows x 4 chunks and lands as four consecutive 64-k tiles of 16 rows.
    const int act3d = (K % kCodeK) == 0 && !gather;
    if (act3d) {
        cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K / 64)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
        cuuint32_t box[3] = {64, 16, 4};
        cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tm_act3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(act), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return MOE_ERR_CUDA;
    } else {
        tm_act3 = tm_act;
    }
    // Scale tiles: [E*N rows][scale bytes a row], boxes of 16 bytes x 128 rows,
    // when the row pitch and the base allow 16-byte TMA rows.  MXFP4: K/32
    // bytes a row, a box covers two code stages.  NVFP4: K/16 bytes a row, a box
    // covers one code stage.  MXFP4 with one scale per 512 k: K/512 bytes a
    // row, loaded by the converter threads.
    const int scale_row = kNv ? K / 16 : K / scale_block;
    const int scale_tma = (kNv || scale_block == 32) && (K % (kNv ? 256 : 512)) == 0 &&
                          (reinterpret_cast<uintptr_t>(scales) & 15) == 0;
    if (scale_tma && swiglu) {
        if (!encode_swiglu_view(&tm_scales, scales, static_cast<cuuint64_t>(scale_row), 16,
                                CU_TENSOR_MAP_SWIZZLE_NONE))
            return MOE_ERR_CUDA;
    } else if (scale_tma) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(scale_row),
                              static_cast<cuuint64_t>(E) * static_cast<cuuint64_t>(N)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(scale_row)};
        cuuint32_t box[2] = {16, 128};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(scales), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return MOE_ERR_CUDA;
    } else {
        tm_scales = tm_codes;
    }
    // Devices (0..63) whose shared-memory attribute is set (one mask per format);
    // others set it on every call.
    static std::atomic<uint64_t> attr_dev_mask{0};   // one per instantiation
    const int smem_bytes = kNv ? kSmemBytesNv : kSmemBytes;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    const uint64_t dev_bit = dev >= 0 && dev < 64 ? 1ull << dev : 0;
    if (!(attr_dev_mask.load(std::memory_order_acquire) & dev_bit) || !dev_bit) {
        const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
        const bool ok =
            kNv ? cudaFuncSetAttribute(grouped_gemm_nvfp4_kernel<true>, a, smem_bytes) == cudaSuccess &&
                      cudaFuncSetAttribute(grouped_gemm_nvfp4_kernel<false>, a, smem_bytes) == cudaSuccess
                : cudaFuncSetAttribute(grouped_gemm_kernel<true, kMap>, a, smem_bytes) == cudaSuccess &&
                      cudaFuncSetAttribute(grouped_gemm_kernel<false, kMap>, a, smem_bytes) == cudaSuccess;
        if (!ok) return MOE_ERR_CUDA;
        if (kMap == kMapNone &&
            (kNv ? cudaFuncSetAttribute(grouped_gemm_nvfp4_pair_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes)
                 : cudaFuncSetAttribute(grouped_gemm_pair_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes)) !=
                cudaSuccess)
            return MOE_ERR_CUDA;
        attr_dev_mask.fetch_or(dev_bit, std::memory_order_release);
    }
    Params p;
    p.scales = scales;
    p.group_sizes = group_sizes;
    p.out = out;
    p.status = status;
    p.rows = rows;
    p.K = K;
    p.N = N;
    p.E = E;
    p.out_bf16 = swiglu ? 1 : out_bf16;
    p.swiglu = swiglu;
    p.I = swiglu ? N / 2 : 0;
    p.h_k8 = h_k8;
    p.allow_wide = act_k8;
    p.n_tiles = swiglu ? (N / 2 + kBN / 2 - 1) / (kBN / 2) : (N + kBN - 1) / kBN;
    p.k_stages = 4 * ((K + kCodeK - 1) / kCodeK);
    p.scale_row = scale_row;
    p.k_blocks = K / 32;
    p.scale_shift = scale_block == 512 ? 4 : 0;
    p.scale_vec2 = ((K / 32) % 2 == 0) && ((reinterpret_cast<uintptr_t>(scales) & 1) == 0);
    p.scale_full = p.scale_vec2 && (K % kCodeK) == 0;
    p.wait_limit_ns = wait_limit_ns;
    p.act_k8 = act_k8;
    p.act3d = act3d;
    p.scale_tma = scale_tma;
    p.gather_slot = gather_slot;
    p.gather_k = gather_k;
    p.act_rows = act_rows;
    p.out_row = out_row;
    // Bands over 32 rows in CTA pairs (each SM then loads half of every
    // activation tile): with K8 activations and an even number of column
    // tiles, when the bands average at least 64 rows (the wide mode's shapes)
    // or when forced, and when the device keeps at least half its SMs' worth
    // of pairs resident (the grid is that many pairs).
    const int pmode = g_pair_mode.load(std::memory_order_relaxed);
    int pair_grid = 0;
    if (kMap == kMapNone && act_k8 && p.n_tiles % 2 == 0 && pmode != 1 &&
        (pmode == 2 || static_cast<long long>(rows) >= 64LL * E)) {
        const int nc = pair_clusters<kNv>(num_sms, smem_bytes);
        if (2 * nc >= num_sms / 2) pair_grid = 2 * (nc < num_sms / 2 ? nc : num_sms / 2);
    }
    // Two launches: bands of 1..32 rows, then bands of 33 or more (a launch
    // whose class has no band returns from its prologue).  The second is a
    // programmatic dependent launch: the two read the same inputs and write
    // disjoint output rows, so its CTAs may start on the SMs the first one's
    // CTAs leave (every kernel here signals its dependents on entry).  The
    // first launch, and whatever follows the second, keep full stream order:
    // the first starts after all earlier work, so the second does too.
    for (int cls = 0; cls < 2; ++cls) {
        p.band_lo = cls == 0 ? 1 : kPartCols + 1;
        p.band_hi = cls == 0 ? kPartCols : INT32_MAX;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = cls == 1 ? 1 : 0;
        cudaError_t err;
        if constexpr (kNv) {
            if (cls == 0) {
                cfg.gridDim = dim3(num_sms);
                err = cudaLaunchKernelEx(&cfg, grouped_gemm_nvfp4_kernel<true>, tm_codes, tm_act, tm_act3,
                                         tm_scales, tm_act64, p, ws2);
            } else if (pair_grid > 0) {
                cfg.gridDim = dim3(pair_grid);
                err = cudaLaunchKernelEx(&cfg, grouped_gemm_nvfp4_pair_kernel, tm_codes, tm_act, tm_act32,
                                         tm_scales, tm_act64, p, ws2);
            } else {
                cfg.gridDim = dim3(num_sms);
                err = cudaLaunchKernelEx(&cfg, grouped_gemm_nvfp4_kernel<false>, tm_codes, tm_act, tm_act32,
                                         tm_scales, tm_act64, p, ws2);
            }
        } else {
            if (cls == 0) {
                cfg.gridDim = dim3(num_sms);
                err = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<true, kMap>, tm_codes, tm_act, tm_act3,
                                         tm_scales, tm_act64, p);
            } else if (pair_grid > 0) {
                cfg.gridDim = dim3(pair_grid);
                err = cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel, tm_codes, tm_act, tm_act32,
                                         tm_scales, tm_act64, p);
            } else {
                cfg.gridDim = dim3(num_sms);
                err = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<false, kMap>, tm_codes, tm_act, tm_act32,
                                         tm_scales, tm_act64, p);
            }
        }
        if (err != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status launch_grouped_gemm(const uint16_t *act, int rows, int K, const uint8_t *codes,
                               const uint8_t *scales, const int32_t *group_sizes, int E, int N,
                               void *out, int out_bf16, int act_k8, int *status,
                               uint64_t wait_limit_ns, cudaStream_t stream, int num_sms) {
    return launch_gemm<false>(act, rows, K, codes, scales, nullptr, group_sizes, E, N, out,
                              out_bf16, act_k8, 0, 0, status, wait_limit_ns, stream, num_sms);
}

moe_status launch_grouped_gemm_block(const uint16_t *act, int rows, int K, int scale_block,
                                     const uint8_t *codes, const uint8_t *scales,
                                     const int32_t *group_sizes, int E, int N, void *out,
                                     int out_bf16, int act_k8, int *status, uint64_t wait_limit_ns,
                                     cudaStream_t stream, int num_sms) {
    return launch_gemm<false>(act, rows, K, codes, scales, nullptr, group_sizes, E, N, out,
                              out_bf16, act_k8, 0, 0, status, wait_limit_ns, stream, num_sms,
                              scale_block);
}

moe_status launch_grouped_gemm_swiglu(const uint16_t *act, int rows, int K, const uint8_t *codes,
                                      const uint8_t *scales, const int32_t *group_sizes, int E,
                                      int N, uint16_t *h, int act_k8, int h_k8, int *status,
                                      uint64_t wait_limit_ns, cudaStream_t stream, int num_sms) {
    return launch_gemm<false>(act, rows, K, codes, scales, nullptr, group_sizes, E, N, h, 1,
                              act_k8, 1, h_k8, status, wait_limit_ns, stream, num_sms);
}

moe_status launch_grouped_gemm_swiglu_gather(const uint16_t *x_k8, int act_rows, int top_k,
                                             const int32_t *sorted_slot, int rows, int K,
                                             const uint8_t *codes, const uint8_t *scales,
                                             const int32_t *group_sizes, int E, int N, uint16_t *h,
                                             int h_k8, int *status, uint64_t wait_limit_ns,
                                             cudaStream_t stream, int num_sms) {
    return launch_gemm<false, gemm::kMapGather>(x_k8, rows, K, codes, scales, nullptr, group_sizes, E, N,
                                          h, 1, 1, 1, h_k8, status, wait_limit_ns, stream, num_sms,
                                          32, sorted_slot, top_k, act_rows, nullptr);
}

moe_status launch_grouped_gemm_scatter(const uint16_t *act, int rows, int K, const uint8_t *codes,
                                       const uint8_t *scales, const int32_t *group_sizes, int E,
                                       int N, const int32_t *out_row, void *out, int out_bf16,
                                       int act_k8, int *status, uint64_t wait_limit_ns,
                                       cudaStream_t stream, int num_sms) {
    return launch_gemm<false, gemm::kMapScatter>(act, rows, K, codes, scales, nullptr, group_sizes, E, N,
                                           out, out_bf16, act_k8, 0, 0, status, wait_limit_ns,
                                           stream, num_sms, 32, nullptr, 1, 0, out_row);
}

moe_status launch_grouped_gemm_nvfp4(const uint16_t *act, int rows, int K, const uint8_t *codes,
                                     const uint8_t *scales16, const float *weight_scale_2,
                                     const int32_t *group_sizes, int E, int N, void *out,
                                     int out_bf16, int act_k8, int *status,
                                     uint64_t wait_limit_ns, cudaStream_t stream, int num_sms) {
    return launch_gemm<true>(act, rows, K, codes, scales16, weight_scale_2, group_sizes, E, N, out,
                             out_bf16, act_k8, 0, 0, status, wait_limit_ns, stream, num_sms);
}

moe_status launch_decode_expert(const uint8_t *codes, const uint8_t *scales, int N, int K, int e,
                                uint16_t *out, int *status, cudaStream_t stream) {
    const long long total = static_cast<long long>(N) * (K / 32);
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    gemm::decode_expert_kernel<<<blocks, 256, 0, stream>>>(codes, scales, N, K, e, out, status);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_bounded_wait(uint64_t limit_ns, int *status, cudaStream_t stream) {
    gemm::bounded_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
