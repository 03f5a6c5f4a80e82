// Allocation-free variant of the schedule-table builder.
//
// Some callers cannot allocate device memory when they need the routing
// tables: serving processes that reserve their whole device-memory budget at
// start-up and forbid any later allocation, and latency-critical loops that
// must not enter cudaMalloc/cudaFree because those calls can synchronise the
// device and stall every stream.  moeffn_schedule_tables_noalloc gives them
// the per-expert counts, 128-row padded offsets and (token, k) -> slot table
// with no workspace argument and no allocation: its scratch lives in one
// file-scope device array that is part of the loaded library image.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the parts that must start at zero are cleared by each call.
// Calls that overlap on the GPU (different streams without ordering, or
// several host threads) race on the array and give wrong tables.
#include "moeffn.h"
#include "common.cuh"

namespace {

using moeffn::DevStatus;
using moeffn::kPoolBlock;

// layout: [0, 64) status words (last-block ticket), [64, 64 + 4N) in-chunk
// ranks, then the per-chunk histograms [ceil(N/1024)][E] (4-byte ints)
static __device__ __align__(256) unsigned char g_sched_scratch[MOEFFN_NOALLOC_SCRATCH_BYTES];

constexpr int kChunk = 1024;

size_t scratch_need(int64_t N, int64_t E) {
    const int64_t nchunks = (N + kChunk - 1) / kChunk;
    return 64 + static_cast<size_t>(4 * N) + static_cast<size_t>(4 * nchunks * E);
}

__device__ int block_scan_1024(int v, int* s_warp, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = s_warp[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        s_warp[lane] = s;
    }
    __syncthreads();
    total = s_warp[31];
    const int r = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
    __syncthreads();
    return r;
}

// One launch: every block ranks its 1024 entries stably per expert and
// writes its histogram; the last block to finish scans the histograms into
// per-chunk bases, writes counts and padded offsets, then every slot.
__global__ void __launch_bounds__(kChunk) sched_tables_noalloc_kernel(
    const int64_t* __restrict__ topk_idx, int N, int E, int* __restrict__ counts,
    int* __restrict__ offsets, int* __restrict__ slots, unsigned char* scratch) {
    extern __shared__ int s_wcnt[];   // [32][E]
    __shared__ int s_warp[32];
    __shared__ int s_last;
    DevStatus* st = reinterpret_cast<DevStatus*>(scratch);
    int* rank = reinterpret_cast<int*>(scratch + 64);
    int* hist = rank + N;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 32 * E; i += kChunk) s_wcnt[i] = 0;
    __syncthreads();
    const int i = blockIdx.x * kChunk + tid;
    int e = -1;
    if (i < N) {
        const int64_t v = topk_idx[i];
        if (v >= 0 && v < E) e = static_cast<int>(v);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rw = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rw == 0) s_wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += kChunk) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int c = s_wcnt[w * E + x];
            s_wcnt[w * E + x] = run;
            run += c;
        }
        hist[static_cast<size_t>(blockIdx.x) * E + x] = run;
    }
    __syncthreads();
    if (i < N) rank[i] = e >= 0 ? s_wcnt[warp * E + e] + rw : -1;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&st->done_counter, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    int cnt = 0;
    if (tid < E) {
        int run = 0;
        for (int c = 0; c < static_cast<int>(gridDim.x); ++c) {
            int* p = hist + static_cast<size_t>(c) * E + tid;
            const int h = __ldcg(p);
            *p = run;
            run += h;
        }
        cnt = run;
        counts[tid] = cnt;
    }
    int total;
    const int off = block_scan_1024(tid < E ? (cnt + kPoolBlock - 1) / kPoolBlock * kPoolBlock : 0, s_warp, total);
    if (tid < E) offsets[tid] = off;
    if (tid == 0) offsets[E] = total;
    __syncthreads();   // offsets (global) visible to the whole block
    for (int j = tid; j < N; j += kChunk) {
        const int64_t v = topk_idx[j];
        int s = -1;
        if (v >= 0 && v < E) {
            const int ee = static_cast<int>(v);
            s = offsets[ee] + __ldcg(hist + static_cast<size_t>(j / kChunk) * E + ee) + __ldcg(rank + j);
        }
        slots[j] = s;
    }
    if (tid == 0) st->done_counter = 0;
}

// Device address of g_sched_scratch on the current device (the host-side
// name of the array is not a device address).  Looked up on every call: once
// the library's module is loaded on the device this is a host-side table
// lookup, and it stays right if the context was torn down and the module
// reloaded at another address.  With lazy module loading (the default since
// CUDA 12.2) the first lookup on a device loads the module, which reserves
// the array; that is why callers make their first call at start-up.
moeffn_status scratch_for_current_device(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sched_scratch) != cudaSuccess || !p) return MOEFFN_ERR_CUDA;
    *out = p;
    return MOEFFN_OK;
}

}  // namespace

extern "C" moeffn_status moeffn_schedule_tables_noalloc(const int64_t* topk_idx, int32_t num_tokens,
                                                        int32_t num_experts, int32_t topk, int32_t* counts,
                                                        int32_t* offsets, int32_t* slots, moeffn_stream stream) {
    if (num_tokens < 0 || num_experts < 1 || num_experts > 1024 || topk < 1 || topk > num_experts || topk > 32)
        return MOEFFN_ERR_INVALID_ARG;
    if (!counts || !offsets) return MOEFFN_ERR_INVALID_ARG;
    const int64_t N = static_cast<int64_t>(num_tokens) * topk;
    if (N > 0 && (!topk_idx || !slots)) return MOEFFN_ERR_INVALID_ARG;
    if (scratch_need(N, num_experts) > MOEFFN_NOALLOC_SCRATCH_BYTES) return MOEFFN_ERR_WORKSPACE_TOO_SMALL;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOEFFN_ERR_CUDA;
    if (major != 10 || minor != 3) return MOEFFN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    moeffn_status s = scratch_for_current_device(&scratch);
    if (s != MOEFFN_OK) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        // no entries: every expert is empty
        if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * num_experts, st) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (num_experts + 1), st) != cudaSuccess)
            return MOEFFN_ERR_CUDA;
        return MOEFFN_OK;
    }
    // the last-block ticket must start at zero on every call
    if (cudaMemsetAsync(scratch, 0, 64, st) != cudaSuccess) return MOEFFN_ERR_CUDA;
    const size_t smem = static_cast<size_t>(32) * num_experts * sizeof(int);
    if (cudaFuncSetAttribute(sched_tables_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             32 * 1024 * static_cast<int>(sizeof(int))) != cudaSuccess)
        return MOEFFN_ERR_CUDA;
    const int nchunks = static_cast<int>((N + kChunk - 1) / kChunk);
    sched_tables_noalloc_kernel<<<nchunks, kChunk, smem, st>>>(topk_idx, static_cast<int>(N), num_experts, counts,
                                                               offsets, slots, static_cast<unsigned char*>(scratch));
    return cudaGetLastError() == cudaSuccess ? MOEFFN_OK : MOEFFN_ERR_CUDA;
}
