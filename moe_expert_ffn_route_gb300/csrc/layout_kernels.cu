// Routing, schedule-table, gather, combine and weight-preparation kernels
// of the fused MoE expert forward (everything except the two grouped GEMMs).
//
// Sources (page titles and sections, in English translation where the page
// is Chinese: the practice page is 通算融合算子（五）：实战, the notes are
// MegaMoE：把 MoE 前向路径压进一个通信计算融合核):
//  - MegaMoE blog 4.2 "Dispatch warps": per-expert counting with block-local
//    atomics over all (token, k) entries, then the pull of each routed
//    token's hidden vector into the expert pool (here a local gather).
//  - "Fused comm/compute operators (5): practice", section 2 "schedule
//    tables": the expert-sorted pool with each expert padded to 128 rows,
//    the padded prefix, the slot table [token][k] shared by scatter (L1) and
//    gather-back (L2), the slack per 128-row block, built by a vectorised
//    GPU builder (one sort + scatter) rather than a host loop.
//  - MegaMoE code-reading notes, "Stage 6: combine": per token, FP32 sum of
//    the BF16 expert outputs of its valid top-k slots, cast back to BF16.
//  - MegaMoE blog 7.3 and the SymmBuffer page section 7 (weight transform:
//    gate/up interleave by 8 rows, scale transpose for tensor-memory copy).
#include "common.cuh"
#include "kernels.h"

#include <cuda_bf16.h>

namespace moeffn {

// ---------------------------------------------------------------------------
// a0: routing.  One warp per token; lane l holds logits l, l+32, ...
// ---------------------------------------------------------------------------
// Unsigned keys in the order of the floats they come from (no NaN, no -0).
__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_order_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

template <int PER_LANE>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int64_t* __restrict__ idx,
                                                         float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const float* l = logits + static_cast<size_t>(t) * E;
    float v[PER_LANE];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = lane + 32 * i;
        // a NaN logit ranks below every number, like -inf: every candidate
        // then compares, and each round picks a valid, untaken expert; -0 is
        // taken as +0 (they compare equal, so ties between them go by index)
        const float x = e < E ? __ldg(l + e) : -INFINITY;
        v[i] = x == x ? x + 0.0f : -INFINITY;
        if (e >= E) taken |= 1u << i;
    }
    float my_v = 0.f;
    int my_e = -1;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = lane + 32 * i;
            if (!((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
                bv = v[i];
                be = e;
            }
        }
        // across the warp: the largest value, then the lowest expert holding it
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, order_key(bv));
        const int win = __reduce_min_sync(0xffffffffu, order_key(bv) == kmax ? be : 0x7FFFFFFF);
        if (win < E && (win & 31) == lane) taken |= 1u << (win >> 5);
        if (lane == j) {
            my_v = from_order_key(kmax);
            my_e = win;
        }
    }
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    float p = lane < k ? expf(my_v - top) : 0.f;
    float s = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane < k) {
        idx[static_cast<size_t>(t) * k + lane] = my_e;
        w[static_cast<size_t>(t) * k + lane] = p / s;
    }
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int64_t* idx, float* w,
                              cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int threads = 256, blocks = (T * 32 + threads - 1) / threads;
    const int per_lane = (E + 31) / 32;
    if (per_lane <= 2)
        route_topk_kernel<2><<<blocks, threads, 0, stream>>>(logits, T, E, k, idx, w);
    else if (per_lane <= 8)
        route_topk_kernel<8><<<blocks, threads, 0, stream>>>(logits, T, E, k, idx, w);
    else
        route_topk_kernel<32><<<blocks, threads, 0, stream>>>(logits, T, E, k, idx, w);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// a1-a3 part 1: per-chunk histograms and stable in-chunk ranks, then (last
// block) the per-expert chunk bases, counts, 128-row padded offsets and the
// token-tile prefix.
// ---------------------------------------------------------------------------
constexpr int kChunk = 1024;   // (token, k) entries per block

__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* s_warp, int& total) {
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
        s_warp[lane] = s;   // inclusive warp totals
    }
    __syncthreads();
    total = s_warp[31];
    const int before = warp > 0 ? s_warp[warp - 1] : 0;
    const int r = before + x - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kChunk) layout_count_kernel(
    const int64_t* __restrict__ topk_idx, int N, int E, int tile_n, int paired, int* __restrict__ hist,
    int* __restrict__ rank, int* __restrict__ counts, int* __restrict__ offsets,
    int* __restrict__ tiles, int* __restrict__ tile_rows, DevStatus* st) {
    extern __shared__ int s_wcnt[];   // [32 warps][E]
    __shared__ int s_warp[32];
    __shared__ int s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 32 * E; i += kChunk) s_wcnt[i] = 0;
    pdl_wait();
    pdl_launch_dependents();
    __syncthreads();

    const int i = blockIdx.x * kChunk + tid;
    int e = -1;
    if (i < N) {
        const int64_t v = topk_idx[i];
        if (v >= 0 && v < E)
            e = static_cast<int>(v);
        else if (v != -1)
            atomicOr(&st->code, DEV_ERR_BAD_EXPERT);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank_in_warp == 0) s_wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    // exclusive scan over the 32 warps for every expert; chunk histogram
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
    if (i < N) rank[i] = e >= 0 ? s_wcnt[warp * E + e] + rank_in_warp : -1;

    // last block to finish turns the chunk histograms into bases and offsets
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&st->done_counter, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int nchunks = gridDim.x;
    int cnt = 0;
    if (tid < E) {
        // chunk c's first rank inside expert tid; eight chunk counts in flight at a time
        int run = 0;
        for (int c0 = 0; c0 < nchunks; c0 += 8) {
            int h[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                h[u] = c0 + u < nchunks ? __ldcg(hist + static_cast<size_t>(c0 + u) * E + tid) : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c0 + u < nchunks) {
                    hist[static_cast<size_t>(c0 + u) * E + tid] = run;
                    run += h[u];
                }
        }
        cnt = run;
        counts[tid] = cnt;
    }
    int total;
    const int padded = tid < E ? (cnt + kPoolBlock - 1) / kPoolBlock * kPoolBlock : 0;
    const int off = block_exclusive_scan_1024(padded, s_warp, total);
    if (tid < E) offsets[tid] = off;
    if (tid == 0) offsets[E] = total;
    // tiles of an expert: as few as tile_n allows (an even number when paired),
    // equal, a multiple of 16 rows
    int ntile = tid < E ? (cnt + tile_n - 1) / tile_n : 0;
    if (paired) ntile += ntile & 1;
    const int toff = block_exclusive_scan_1024(ntile, s_warp, total);
    if (tid < E) {
        tiles[tid] = toff;
        const int per = ntile ? (cnt + ntile - 1) / ntile : kTileQuantum;
        tile_rows[tid] = (per + kTileQuantum - 1) / kTileQuantum * kTileQuantum;
    }
    if (tid == 0) {
        tiles[E] = total;
        st->done_counter = 0;   // ready for the next forward on this workspace
    }
}

constexpr int kDispatchSplit = 4;   // warps per token row in the gather (divides 8)

// ---------------------------------------------------------------------------
// a3 part 2 + a4: slots, inverse map, pool weights, and the gather of token
// rows and their scales into the expert-sorted pool.  Blocks [0, nb_tok) take
// 8 / kDispatchSplit tokens each (kDispatchSplit warps per token); the
// remaining blocks fill the padding rows of one expert each.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) dispatch_kernel(
    const uint8_t* __restrict__ x, const uint32_t* __restrict__ x_sf,
    const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int T, int H, int E,
    int k, const int* __restrict__ hist, const int* __restrict__ rank,
    const int* __restrict__ counts, const int* __restrict__ offsets,
    const int* __restrict__ tiles, const int* __restrict__ tile_rows, int* __restrict__ tile_rec,
    int* __restrict__ l1_done, int* __restrict__ slots, int* __restrict__ row2tk,
    float* __restrict__ wpool, int* __restrict__ slack, uint8_t* __restrict__ xpool,
    uint32_t* __restrict__ xpool_sf, int nb_tok, int P_max, int NT_max, DevStatus* st) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();
    pdl_launch_dependents();
    if (static_cast<int>(blockIdx.x) >= nb_tok) {
        // padding rows, slack and the tile records of expert e
        const int e = blockIdx.x - nb_tok;
        const int n = counts[e], beg = offsets[e], end = offsets[e + 1];
        const int t0 = tiles[e], t1 = tiles[e + 1];
        // the GEMM's pool rows and tile indices come from these records: its rows
        // lie in [beg, beg + n) within [beg, end), its tiles in [t0, t1); the
        // block checks the non-empty ranges here, all threads alike
        if (end > beg && (!in_bounds(st, end - 1, P_max, 1) || !in_bounds(st, beg + n, end + 1, 1))) return;
        if (t1 > t0 && !in_bounds(st, t1 - 1, NT_max, 2)) return;
        for (int tt = t0 + threadIdx.x; tt < t1; tt += blockDim.x) {
            if (!in_bounds(st, tt, NT_max, 2)) break;
            int4* rec = reinterpret_cast<int4*>(tile_rec) + 2 * tt;
            rec[0] = make_int4(e, t0, t1 - t0, tile_rows[e]);
            rec[1] = make_int4(beg, n, 0, 0);
            l1_done[tt] = 0;    // counts the L1 epilogue warps that published this tile's rows
        }
        for (int r = beg + n + threadIdx.x; r < end; r += blockDim.x) {
            if (!in_bounds(st, r, P_max, 3)) break;
            row2tk[r] = -1;
            wpool[r] = 0.f;
        }
        for (int b = beg / kPoolBlock + threadIdx.x; b < end / kPoolBlock; b += blockDim.x) {
            if (!in_bounds(st, b, P_max / kPoolBlock, 4)) break;
            const int real = min(kPoolBlock, max(0, n - (b * kPoolBlock - beg)));
            slack[b] = kPoolBlock - real;
        }
        return;
    }
    // kDispatchSplit warps per token, each copying every kDispatchSplit-th
    // 2 KB of the row (enough warps in flight for an HBM-bound copy)
    const int part = warp % kDispatchSplit;
    const int t = blockIdx.x * (8 / kDispatchSplit) + warp / kDispatchSplit;
    if (t >= T) return;
    const int Kb = H / 128;
    // lane j < k resolves entry (t, j)
    int slot = -1, chunk = -1, word = 0;
    if (lane < k) {
        const int i = t * k + lane;
        const int64_t v = topk_idx[i];
        if (v >= 0 && v < E) {
            const int e = static_cast<int>(v);
            const int r = hist[static_cast<size_t>(i / kChunk) * E + e] + rank[i];
            slot = offsets[e] + r;
            const int rows = tile_rows[e];
            chunk = tiles[e] + r / rows;
            if (!in_bounds(st, slot, P_max, 5) || !in_bounds(st, chunk, NT_max, 6)) slot = chunk = -1;
            const int rt = r % rows;
            // 128-row half of the tile, then word 4 l + c for row 32 c + l of that half
            word = (rt >> 7) * 128 + (rt & 31) * 4 + ((rt & 127) >> 5);
            if (part == 0 && slot >= 0) {
                row2tk[slot] = i;
                wpool[slot] = topk_w[i];
            }
        }
        if (part == 0) slots[i] = slot;
    }
    // scales: word kb of the token's row goes to chunk `chunk`, K block kb
    for (int j = 0; j < k; ++j) {
        const int s = __shfl_sync(0xffffffffu, slot, j);
        const int c = __shfl_sync(0xffffffffu, chunk, j);
        const int wd = __shfl_sync(0xffffffffu, word, j);
        if (s < 0) continue;
        for (int kb = lane + 32 * part; kb < Kb; kb += 32 * kDispatchSplit)
            xpool_sf[(static_cast<size_t>(c) * Kb + kb) * 256 + wd] = x_sf[static_cast<size_t>(t) * Kb + kb];
    }
    // token row: read once, write to each valid slot (16-byte vectors)
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    const int nv = H / 16;
    for (int base = 128 * part; base < nv; base += 128 * kDispatchSplit) {
        uint4 buf[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int vi = base + u * 32 + lane;
            if (vi < nv) buf[u] = __ldg(src + vi);
        }
        for (int j = 0; j < k; ++j) {
            const int s = __shfl_sync(0xffffffffu, slot, j);
            if (s < 0) continue;
            uint4* dst = reinterpret_cast<uint4*>(xpool + static_cast<size_t>(s) * H);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int vi = base + u * 32 + lane;
                if (vi < nv) dst[vi] = buf[u];
            }
        }
    }
}

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t stream) {
    const int N = a.T * a.k;
    const int nchunks = (N + kChunk - 1) / kChunk;
    const size_t smem = static_cast<size_t>(32) * a.E * sizeof(int);
    if (smem > 48 * 1024) {
        // per device and cheap: set on every launch that needs more than the default
        cudaError_t err = cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
        if (err != cudaSuccess) return err;
    }
    cudaError_t err = launch_pdl(layout_count_kernel, dim3(nchunks), dim3(kChunk), smem, stream, a.topk_idx, N,
                                 a.E, a.tile_n, a.paired, a.hist, a.rank, a.counts, a.offsets, a.tiles, a.tile_rows,
                                 a.status);
    if (err != cudaSuccess) return err;
    const int tok_per_block = 8 / kDispatchSplit;
    const int nb_tok = (a.T + tok_per_block - 1) / tok_per_block;
    return launch_pdl(dispatch_kernel, dim3(nb_tok + a.E), dim3(256), 0, stream, a.x, a.x_sf, a.topk_idx,
                      a.topk_w, a.T, a.H, a.E, a.k, a.hist, a.rank, a.counts, a.offsets, a.tiles, a.tile_rows,
                      a.tile_rec, a.l1_done, a.slots, a.row2tk, a.wpool, a.slack, a.xpool, a.xpool_sf, nb_tok,
                      a.P_max, a.NT_max, a.status);
}

// ---------------------------------------------------------------------------
// a9: combine.  One block per token; FP32 sum of the BF16 slot rows in j
// order, rounded to BF16.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) combine_kernel(const uint16_t* __restrict__ ypool,
                                                      const int* __restrict__ slots, int H, int k,
                                                      uint16_t* __restrict__ y, int P_max, DevStatus* st) {
    __shared__ int s_slot[32];
    const int t = blockIdx.x;
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x < k) {
        const int s = slots[static_cast<size_t>(t) * k + threadIdx.x];
        s_slot[threadIdx.x] = s < 0 || in_bounds(st, s, P_max, 7) ? s : -1;
    }
    __syncthreads();
    const int nv = H / 8;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        for (int j0 = 0; j0 < k; j0 += 8) {
            // up to 8 slot rows in flight at once, then summed in j order
            uint4 q[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int s = j0 + jj < k ? s_slot[j0 + jj] : -1;
                q[jj] = s >= 0 ? __ldg(reinterpret_cast<const uint4*>(ypool + static_cast<size_t>(s) * H) + v)
                               : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                if (j0 + jj >= k || s_slot[j0 + jj] < 0) continue;
                const uint32_t w[4] = {q[jj].x, q[jj].y, q[jj].z, q[jj].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] += __uint_as_float(w[i] << 16);
                    acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
                }
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
            o[i] = *reinterpret_cast<const uint32_t*>(&p);
        }
        reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * H)[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

cudaError_t launch_combine(const uint16_t* ypool, const int* slots, int T, int H, int k,
                           uint16_t* y, int P_max, DevStatus* status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(combine_kernel, dim3(T), dim3(128), 0, stream, ypool, slots, H, k, y, P_max, status);
}

// ---------------------------------------------------------------------------
// weight preparation: W1 rows regrouped so that each 128-row block holds
// gate and up of 64 consecutive channels in bands of 32 (gate c0..c0+31,
// up c0..c0+31, gate c0+32..c0+63, up c0+32..c0+63), undoing the boundary's
// interleave by 8; W2 copied; scales of both re-laid per 128-row block and
// 128-wide K block into the tensor-memory copy order (word 4*l + c = row
// 32*c + l).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int w1_source_row(int p, int I) {
    (void)I;
    const int band = (p % 128) / 32;             // 0 gate lo, 1 up lo, 2 gate hi, 3 up hi
    const int c = 64 * (p / 128) + 32 * (band >> 1) + (p % 32);
    return 16 * (c / 8) + (c % 8) + ((band & 1) ? 8 : 0);
}

__global__ void prepare_rows_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                    int rows_per_expert, int row_bytes, int I, int is_w1) {
    const int p = blockIdx.x;                 // destination row within expert
    const int e = blockIdx.y;
    const int r = is_w1 ? w1_source_row(p, I) : p;
    const uint4* s = reinterpret_cast<const uint4*>(src + (static_cast<size_t>(e) * rows_per_expert + r) * row_bytes);
    uint4* d = reinterpret_cast<uint4*>(dst + (static_cast<size_t>(e) * rows_per_expert + p) * row_bytes);
    for (int v = threadIdx.x; v < row_bytes / 16; v += blockDim.x) d[v] = __ldg(s + v);
}

__global__ void prepare_sf_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst,
                                  int rows_per_expert, int kb_per_row, int I, int is_w1) {
    // one block per (expert, 128-row block); threads over (kb, word)
    const int rb = blockIdx.x, e = blockIdx.y;
    const int nblk = rows_per_expert / 128;
    for (int i = threadIdx.x; i < kb_per_row * 128; i += blockDim.x) {
        const int kb = i / 128, wd = i % 128;
        const int l = wd / 4, c = wd % 4;
        const int p = rb * 128 + 32 * c + l;
        const int r = is_w1 ? w1_source_row(p, I) : p;
        dst[((static_cast<size_t>(e) * nblk + rb) * kb_per_row + kb) * 128 + wd] =
            src[(static_cast<size_t>(e) * rows_per_expert + r) * kb_per_row + kb];
    }
}

cudaError_t launch_prepare(const PrepareArgs& a, cudaStream_t stream) {
    const int H = a.H, I = a.I, E = a.E;
    prepare_rows_kernel<<<dim3(2 * I, E), 128, 0, stream>>>(a.w1, a.w1p, 2 * I, H / 2, I, 1);
    prepare_rows_kernel<<<dim3(H, E), 128, 0, stream>>>(a.w2, a.w2p, H, I / 2, I, 0);
    prepare_sf_kernel<<<dim3(2 * I / 128, E), 256, 0, stream>>>(a.w1_sf, a.w1p_sf, 2 * I, H / 128, I, 1);
    prepare_sf_kernel<<<dim3(H / 128, E), 256, 0, stream>>>(a.w2_sf, a.w2p_sf, H, I / 128, I, 0);
    return cudaGetLastError();
}

}  // namespace moeffn
