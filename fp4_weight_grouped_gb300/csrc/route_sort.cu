// Stable counting sort of routing slots into expert row bands, plus the
// activation permutation ("Running DeepSeek V4 Flash on TPU v6", section 1:
// tokens are sorted by expert so the activations form one band of rows per
// expert; the timing note there names the activation permutation as its own
// step).
//
// Three kernels, no atomics on data (results are identical run to run):
//  1. count   — one 1024-slot chunk per block.  Each warp finds equal experts
//               among its 32 slots with __match_any_sync; the rank inside the
//               warp is a popcount; per-warp counts in shared memory are
//               scanned across the 32 warps, giving each slot its rank inside
//               the chunk and each chunk its per-expert total.
//  2. scan    — one block: per expert, exclusive scan of the chunk totals in
//               chunk order; then an exclusive scan over experts (offsets).
//  3. scatter — one warp per slot: row = offset[e] + chunk base + rank; writes
//               both maps and copies the token row (16-byte vectors).
// Scratch (caller workspace): chunk totals [chunks, E] and ranks [rows].
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"
#include "mxfp4_decode.cuh"

namespace moe {
namespace rs {

constexpr int kChunk = 1024;

__global__ void __launch_bounds__(kChunk)
count_kernel(const int32_t *ids, int rows, int E, int32_t *chunk_tot, int32_t *rank, int *status) {
    extern __shared__ uint16_t whist[];   // [32 warps][E]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 32 * E; i += kChunk) whist[i] = 0;
    __syncthreads();
    const int s = blockIdx.x * kChunk + tid;
    int e = -1;
    if (s < rows) {
        e = ids[s];
        if (e < 0 || e >= E) {
            set_status(status, MOE_ERR_DATA);
            e = -2;
        }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank_w == 0) whist[warp * E + e] = static_cast<uint16_t>(__popc(peers));
    __syncthreads();
    for (int x = tid; x < E; x += kChunk) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int c = whist[w * E + x];
            whist[w * E + x] = static_cast<uint16_t>(run);
            run += c;
        }
        chunk_tot[static_cast<size_t>(blockIdx.x) * E + x] = run;
    }
    __syncthreads();
    if (e >= 0) rank[s] = whist[warp * E + e] + rank_w;
}

__global__ void __launch_bounds__(1024)
scan_kernel(int32_t *chunk_tot, int n_chunks, int E, int32_t *group_sizes, int32_t *offsets) {
    __shared__ int warp_tot[32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < E; base += 1024) {
        const int e = base + tid;
        int total = 0;
        if (e < E) {
            for (int c = 0; c < n_chunks; ++c) {
                const int v = chunk_tot[static_cast<size_t>(c) * E + e];
                chunk_tot[static_cast<size_t>(c) * E + e] = total;
                total += v;
            }
            group_sizes[e] = total;
        }
        int incl = total;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = warp_tot[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, w, d);
                if (lane >= d) w += v;
            }
            warp_tot[lane] = w;   // inclusive over warps
        }
        __syncthreads();
        const int before = carry + (warp > 0 ? warp_tot[warp - 1] : 0);
        if (e < E) offsets[e] = before + incl - total;
        __syncthreads();
        if (tid == 0) carry += warp_tot[31];
        __syncthreads();
    }
    if (tid == 0) offsets[E] = carry;
}

// One warp copies a row of `hidden` bf16 (16-byte vectors), optionally into the
// K8-interleaved order (a permutation inside each 16 bytes).
__device__ __forceinline__ void copy_row(const uint16_t *src_row, uint16_t *dst_row, int hidden,
                                         int k8, int lane) {
    const uint4 *src = reinterpret_cast<const uint4 *>(src_row);
    uint4 *dst = reinterpret_cast<uint4 *>(dst_row);
    const int nvec = hidden / 8;
    int i = lane;
    if (k8) {
        for (; i + 96 < nvec; i += 128) {   // four independent 16-byte loads in flight
            const uint4 a = __ldg(src + i), b = __ldg(src + i + 32), c = __ldg(src + i + 64),
                        d = __ldg(src + i + 96);
            dst[i] = interleave8(a);
            dst[i + 32] = interleave8(b);
            dst[i + 64] = interleave8(c);
            dst[i + 96] = interleave8(d);
        }
        for (; i < nvec; i += 32) dst[i] = interleave8(__ldg(src + i));
    } else {
        for (; i + 96 < nvec; i += 128) {
            const uint4 a = __ldg(src + i), b = __ldg(src + i + 32), c = __ldg(src + i + 64),
                        d = __ldg(src + i + 96);
            dst[i] = a;
            dst[i + 32] = b;
            dst[i + 64] = c;
            dst[i + 96] = d;
        }
        for (; i < nvec; i += 32) dst[i] = __ldg(src + i);
    }
}

// One warp per routing slot s: its sorted row, and the activation copies.
// x_sorted (gather): row `row` <- x[s / k].  x_tok (token order, K8): the warp
// of slot t*k copies x[t], once per token and whatever its ids.
__global__ void __launch_bounds__(256)
scatter_kernel(const int32_t *ids, int rows, int k, int E, const int32_t *chunk_base,
               const int32_t *offsets, const int32_t *rank, int32_t *sorted_slot,
               int32_t *slot_to_row, const uint16_t *x, int hidden, uint16_t *x_sorted, int x_k8,
               uint16_t *x_tok) {
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (s >= rows) return;
    if (x_tok && s % k == 0)
        copy_row(x + static_cast<size_t>(s / k) * hidden, x_tok + static_cast<size_t>(s / k) * hidden,
                 hidden, 1, lane);
    const int e = ids[s];
    if (e < 0 || e >= E) {                 // recorded by the count kernel
        if (lane == 0) slot_to_row[s] = -1;   // no row: the combine skips this slot
        return;
    }
    const int row =
        offsets[e] + chunk_base[static_cast<size_t>(s / kChunk) * E + e] + rank[s];
    if (lane == 0) {
        sorted_slot[row] = s;
        slot_to_row[s] = row;
    }
    if (x_sorted)
        copy_row(x + static_cast<size_t>(s / k) * hidden, x_sorted + static_cast<size_t>(row) * hidden,
                 hidden, x_k8, lane);
}

}  // namespace rs

size_t route_sort_scratch_bytes(int T, int k, int E) {
    const size_t rows = static_cast<size_t>(T) * k;
    const size_t chunks = (rows + rs::kChunk - 1) / rs::kChunk;
    auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    return up(chunks * E * 4) + up(rows * 4);
}

moe_status launch_route_sort(const int32_t *ids, int T, int k, int E, int32_t *group_sizes,
                             int32_t *offsets, int32_t *sorted_slot, int32_t *slot_to_row,
                             const uint16_t *x, int hidden, uint16_t *x_sorted, int x_k8,
                             void *scratch, int *status, cudaStream_t stream, int *launches,
                             uint16_t *x_tok) {
    const int rows = T * k;
    const int chunks = (rows + rs::kChunk - 1) / rs::kChunk;
    auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    int32_t *chunk_tot = reinterpret_cast<int32_t *>(scratch);
    int32_t *rank = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(scratch) +
                                                up(static_cast<size_t>(chunks) * E * 4));
    *launches = 0;
    if (chunks > 0) {
        const size_t shmem = static_cast<size_t>(32) * E * sizeof(uint16_t);
        // Devices (0..63) whose shared-memory attribute is set; others set it on every call.
        static std::atomic<uint64_t> attr_dev_mask{0};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
        const uint64_t dev_bit = dev >= 0 && dev < 64 ? 1ull << dev : 0;
        if (!(attr_dev_mask.load(std::memory_order_acquire) & dev_bit) || !dev_bit) {
            if (cudaFuncSetAttribute(rs::count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     32 * 1024 * 2) != cudaSuccess)
                return MOE_ERR_CUDA;
            attr_dev_mask.fetch_or(dev_bit, std::memory_order_release);
        }
        rs::count_kernel<<<chunks, rs::kChunk, shmem, stream>>>(ids, rows, E, chunk_tot, rank,
                                                               status);
        ++*launches;
    }
    rs::scan_kernel<<<1, 1024, 0, stream>>>(chunk_tot, chunks, E, group_sizes, offsets);
    ++*launches;
    if (rows > 0) {
        rs::scatter_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(ids, rows, k, E, chunk_tot, offsets,
                                                               rank, sorted_slot, slot_to_row, x,
                                                               hidden, x_sorted, x_k8, x_tok);
        ++*launches;
    }
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Fixed-capacity variant: the same three kernels with their scratch in static
// device storage, for callers that cannot allocate or pass a workspace at the
// point of the call.  Layout of the array: the status word in the first 256
// bytes, then the scratch exactly as launch_route_sort lays it out.  The
// chunk totals and ranks are written in full before they are read; only the
// status word needs clearing, which every call does on its stream.

constexpr size_t kNoAllocStatusBytes = 256;

static __device__ __align__(256) uint8_t
    noalloc_area[kNoAllocStatusBytes + MOE_ROUTE_SORT_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex noalloc_mutex;
// Device address of noalloc_area per device, with the context it was looked up
// in: after a device reset the primary context (and the module holding the
// array) is created anew, so the address is looked up again.
void *noalloc_base[kMaxDevices];
CUcontext noalloc_ctx[kMaxDevices];

CUcontext current_context() {
    using Fn = CUresult (*)(CUcontext *);
    static const Fn fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<Fn>(nullptr);
        return reinterpret_cast<Fn>(ptr);
    }();
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}
}  // namespace

moe_status launch_route_sort_noalloc(const int32_t *ids, int T, int k, int E,
                                     int32_t *group_sizes, int32_t *offsets,
                                     int32_t *sorted_slot, int32_t *slot_to_row,
                                     const uint16_t *x, int hidden, uint16_t *x_sorted, int x_k8,
                                     cudaStream_t stream, int *launches) {
    *launches = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(noalloc_mutex);
        // A thread whose context is not yet current (null) or differs from the
        // one of the lookup looks the address up again; the lookup itself makes
        // the device's primary context current.
        if (!noalloc_base[dev] || current_context() != noalloc_ctx[dev]) {
            noalloc_base[dev] = nullptr;
            if (cudaGetSymbolAddress(&noalloc_base[dev], noalloc_area) != cudaSuccess) {
                noalloc_base[dev] = nullptr;
                return MOE_ERR_CUDA;
            }
            noalloc_ctx[dev] = current_context();
        }
        base = noalloc_base[dev];
    }
    int *status = static_cast<int *>(base);
    if (cudaMemsetAsync(status, 0, sizeof(int), stream) != cudaSuccess) return MOE_ERR_CUDA;
    return launch_route_sort(ids, T, k, E, group_sizes, offsets, sorted_slot, slot_to_row, x,
                             hidden, x_sorted, x_k8,
                             static_cast<uint8_t *>(base) + kNoAllocStatusBytes, status, stream,
                             launches);
}

}  // namespace moe
