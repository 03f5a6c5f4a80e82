// Grouped GEMMs of the fused MoE expert forward on 5th-generation tensor
// cores (tcgen05, sm_103a): block-scaled E2M1 weights x E4M3 tokens with
// UE8M0 per-32 scales, FP32 accumulation in tensor memory.
//
//   L1:  Z_e = X_e W1_e^T  (per expert, rows of the expert-sorted pool)
//        epilogue: g, u <- bf16(Z gate, Z up); h = silu(g) * u * w_topk;
//        per row and 32 channels: amax -> UE8M0 exponent -> E4M3 codes
//   L2:  Y_e = H_e W2_e^T, epilogue: BF16 rows of the output pool
//
// Sources: MegaMoE code-reading notes, "Stage 3: FP8 x FP4 two-layer GEMM"
// (layer equations, formats, weights in the MMA's first operand and tokens
// in the second -- "swap A/B"), "Stage 4: SwiGLU and requantisation in the
// L1 epilogue", "TMA loads and the UMMA pipeline" (multi-stage full/empty
// barriers), "TMEM column allocation" (two accumulators plus scale-factor
// columns); MegaMoE blog 4.5 "MMA issue" (4 MMAs of K = 32 per 128-wide K
// block, one scale byte selected per MMA) and 4.6 "Epilogue warps".
//
// GB300 design (not the pages' SM100 kernel): one persistent CTA per SM,
// 6 warps -- warp 0 issues TMA, warp 1 issues tcgen05.cp/mma from one
// thread, warps 2..5 drain TMEM.  A tile is two 128-row weight tiles (L1:
// the gate and the up rows of the same 128 channels; L2: 256 output
// channels) against one token tile of tile_n rows, so each thread of the
// epilogue holds gate and up of one channel for every token of the tile.
// Token tiles never straddle experts; scale factors of a token tile are
// stored per tile in tensor-memory copy order, so every stage loads one
// 512-byte scale chunk per operand.
#include "common.cuh"
#include "kernels.h"

#include <cuda_bf16.h>

namespace moeffn {

template <int BN>
struct GemmCfg {
    static constexpr int A_BYTES = 128 * 128;     // 128 weight rows x 128 K (E2M1, 16-byte padded)
    // A TMA load of packed E2M1 (16U4_ALIGN16B) signals the packed global
    // bytes as its transaction count although it fills A_BYTES of shared memory
    static constexpr int A_TX_BYTES = A_BYTES / 2;
    static constexpr int B_BYTES = BN * 128;      // BN token rows x 128 K (E4M3)
    static constexpr int SF_BYTES = 2048;         // SFA0 | SFA1 | SFB (512 each) | pad
    static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES + SF_BYTES;
    static constexpr int EPI_BYTES = 4 * 32 * 33 * 4;   // per-warp 32x33 float transpose
    static constexpr int ACC = BN <= 96 ? 2 : 1;        // accumulator stages in TMEM
    static constexpr int TMEM_NEED = ACC * 2 * BN + 12;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128
                                     : TMEM_NEED <= 256 ? 256 : 512;
    static constexpr int SFA0_COL = ACC * 2 * BN;
    static constexpr int SFA1_COL = SFA0_COL + 4;
    static constexpr int SFB_COL = SFA0_COL + 8;
    static constexpr int MAX_SMEM = 232448;             // 227 KB opt-in per block
    static constexpr int FIXED = EPI_BYTES + 1024 + 256;
    static constexpr int STAGES_FIT = (MAX_SMEM - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int SMEM = FIXED + STAGES * STAGE_BYTES;
    static_assert(TMEM_NEED <= 512, "tensor memory overflow");
    static_assert(STAGES >= 2, "pipeline too shallow");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 128, "token tile");
};

struct TileInfo {
    int e, cb, tile_idx, row0, nvalid;
};

__device__ __forceinline__ TileInfo decode_tile(int t, int ncb, const GemmArgs& p) {
    int lo = 0, hi = p.E;   // tiles[lo]*ncb <= t < tiles[hi]*ncb
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.tiles + mid) * ncb <= t) lo = mid; else hi = mid;
    }
    TileInfo ti;
    const int t0 = __ldg(p.tiles + lo);
    const int ntb = __ldg(p.tiles + lo + 1) - t0;
    const int local = t - t0 * ncb;
    ti.e = lo;
    ti.cb = local / ntb;
    const int nb = local - ti.cb * ntb;
    ti.tile_idx = t0 + nb;
    ti.row0 = __ldg(p.offsets + lo) + nb * p.tile_n;
    ti.nvalid = min(p.tile_n, __ldg(p.counts + lo) - nb * p.tile_n);
    return ti;
}

template <int LAYER, int BN>
__global__ void __launch_bounds__(192, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmArgs p) {
    using C = GemmCfg<BN>;
    constexpr int S = C::STAGES, ACC = C::ACC;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);
    float* epi = reinterpret_cast<float*>(gbase + S * C::STAGE_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + S * C::STAGE_BYTES + C::EPI_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };
    auto tfull = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto tempty = [&](int a) { return bar0 + 8u * (2 * S + ACC + a); };
    const uint32_t mma_done = bar0 + 8u * (2 * S + 2 * ACC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2 * ACC + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < ACC; ++a) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), 128);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int ncb = LAYER == 1 ? p.I / 128 : (p.H + 255) / 256;   // weight-row blocks per expert
    const int nkb = LAYER == 1 ? p.H / 128 : p.I / 128;           // 128-wide K blocks
    const int a_rows = LAYER == 1 ? 2 * p.I : p.H;                 // weight rows per expert
    const int total = __ldg(p.tiles + p.E) * ncb;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            const bool starve = LAYER == 1 && (p.debug_flags & 1);
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile(t, ncb, p);
                const int a0 = ti.e * a_rows + ti.cb * (LAYER == 1 ? 128 : 256);
                const int a1 = a0 + (LAYER == 1 ? p.I : 128);
                const bool a1_valid = LAYER == 1 || (ti.cb * 256 + 128 < p.H);
                const uint8_t* sfa0 = p.sfa + static_cast<size_t>(a0 / 128) * nkb * 512;
                const uint8_t* sfa1 = p.sfa + static_cast<size_t>(a1 / 128) * nkb * 512;
                const uint8_t* sfb = p.sfb + static_cast<size_t>(ti.tile_idx) * nkb * 512;
                const uint32_t bytes = C::A_TX_BYTES + C::B_BYTES + 1024 + (a1_valid ? C::A_TX_BYTES + 512 : 0);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, p.timeout_ns, p.status, 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sb = sbase + stage * C::STAGE_BYTES;
                    const uint32_t sf = sb + 2 * C::A_BYTES + C::B_BYTES;
                    if (!(starve && t == static_cast<int>(blockIdx.x) && kb == 0)) {
                        mbar_arrive_expect_tx(full(stage), bytes);
                        tma_load_2d(sb, &tmA, full(stage), kb * 128, a0);
                        if (a1_valid) tma_load_2d(sb + C::A_BYTES, &tmA, full(stage), kb * 128, a1);
                        tma_load_2d(sb + 2 * C::A_BYTES, &tmB, full(stage), kb * 128, ti.row0);
                        bulk_load(sf, sfa0 + kb * 512, 512, full(stage));
                        if (a1_valid) bulk_load(sf + 512, sfa1 + kb * 512, 512, full(stage));
                        bulk_load(sf + 1024, sfb + kb * 512, 512, full(stage));
                        ++armed[stage];
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // never leave copies in flight into shared memory: wait for the last
            // arming of every stage to land (immediate on the normal path)
            for (int s = 0; s < S; ++s)
                if (armed[s])
                    mbar_wait_bounded(full(s), (armed[s] - 1u) & 1u, abort_flag, p.timeout_ns, p.status, 5, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_mx_e2m1_e4m3(128, BN);
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
                const TileInfo ti = decode_tile(t, ncb, p);
                const bool a1_valid = LAYER == 1 || (ti.cb * 256 + 128 < p.H);
                const int as = it % ACC;
                const uint32_t ap = static_cast<uint32_t>(it / ACC) & 1u;
                if (!mbar_wait_bounded(tempty(as), ap ^ 1u, abort_flag, p.timeout_ns, p.status, 2)) break;
                tc_fence_after();
                const uint32_t d0 = tmem + static_cast<uint32_t>(as * 2 * BN);
                const uint32_t d1 = d0 + BN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(full(stage), phase, abort_flag, p.timeout_ns, p.status, 3)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sb = sbase + stage * C::STAGE_BYTES;
                    const uint32_t sbb = sb + 2 * C::A_BYTES;
                    const uint32_t sf = sbb + C::B_BYTES;
                    tc_cp_sf(tmem + C::SFA0_COL, desc_sf_block(sf));
                    if (a1_valid) tc_cp_sf(tmem + C::SFA1_COL, desc_sf_block(sf + 512));
                    tc_cp_sf(tmem + C::SFB_COL, desc_sf_block(sf + 1024));
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t idesc = IDESC | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
                        const uint64_t bdesc = desc_kmajor_sw128(sbb + 32 * k);
                        const uint32_t acc = (kb | k) != 0;
                        tc_mma_mx(d0, desc_kmajor_sw128(sb + 32 * k), bdesc, idesc, tmem + C::SFA0_COL,
                                  tmem + C::SFB_COL, acc);
                        if (a1_valid)
                            tc_mma_mx(d1, desc_kmajor_sw128(sb + C::A_BYTES + 32 * k), bdesc, idesc,
                                      tmem + C::SFA1_COL, tmem + C::SFB_COL, acc);
                    }
                    tc_commit(empty(stage));
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit(tfull(as));
            }
            // every MMA issued by this thread is complete before TMEM is freed
            tc_commit(mma_done);
            mbar_wait_bounded(mma_done, 0, abort_flag, p.timeout_ns, p.status, 6, false);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                      // TMEM lane quarter of this warp
        float* tb = epi + (warp - 2) * 32 * 33;
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const TileInfo ti = decode_tile(t, ncb, p);
            const int as = it % ACC;
            const uint32_t ap = static_cast<uint32_t>(it / ACC) & 1u;
            const bool got = mbar_wait_bounded(tfull(as), ap, abort_flag, p.timeout_ns, p.status, 4);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(as * 2 * BN);
            for (int j = 0; j < BN / 32; ++j) {
                if (32 * j >= ti.nvalid) break;
                const int rloc = 32 * j + lane;
                const bool valid = rloc < ti.nvalid;
                const int row = ti.row0 + rloc;
                if constexpr (LAYER == 1) {
                    float g[32], u[32];
                    tmem_ld32(tbase + 32 * j, g);
                    tmem_ld32(tbase + BN + 32 * j, u);
                    if (p.debug_flags & 2) {
                        // test hook: raw FP32 accumulators, [P_max][gate I | up I] floats
                        float* zd = reinterpret_cast<float*>(p.ypool);
                        const int c = ti.cb * 128 + 32 * q + lane;
                        for (int n = 0; n < 32 && 32 * j + n < ti.nvalid; ++n) {
                            const size_t r = static_cast<size_t>(ti.row0 + 32 * j + n) * 2 * p.I;
                            zd[r + c] = g[n];
                            zd[r + p.I + c] = u[n];
                        }
                    }
                    const float wv = valid ? __ldg(p.wpool + row) : 0.f;
#pragma unroll
                    for (int n = 0; n < 32; ++n) {
                        const float wn = __shfl_sync(0xffffffffu, wv, n);
                        const float gb = bf16_round(g[n]);
                        const float ub = bf16_round(u[n]);
                        tb[n * 33 + lane] = (gb / (1.0f + expf(-gb))) * ub * wn;
                    }
                    __syncwarp();
                    float v[32];
                    float amax = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        v[i] = tb[lane * 33 + i];
                        amax = fmaxf(amax, fabsf(v[i]));
                    }
                    __syncwarp();
                    const int ex = requant_exponent(amax);
                    const float s = exp2_neg(ex);
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pk[i] = e4m3x2(v[4 * i] * s, v[4 * i + 1] * s) |
                                (e4m3x2(v[4 * i + 2] * s, v[4 * i + 3] * s) << 16);
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(p.hpool + static_cast<size_t>(row) * p.I + ti.cb * 128 + 32 * q);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        const size_t wd = (static_cast<size_t>(ti.tile_idx) * (p.I / 128) + ti.cb) * 128 +
                                          (rloc & 31) * 4 + (rloc >> 5);
                        p.hpool_sf[wd * 4 + q] = static_cast<uint8_t>(ex + 127);
                    }
                } else {
                    const bool a1_valid = ti.cb * 256 + 128 < p.H;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        if (half == 1 && !a1_valid) break;
                        float yv[32];
                        tmem_ld32(tbase + half * BN + 32 * j, yv);
#pragma unroll
                        for (int n = 0; n < 32; ++n) tb[n * 33 + lane] = yv[n];
                        __syncwarp();
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(tb[lane * 33 + 2 * i], tb[lane * 33 + 2 * i + 1]);
                            pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        __syncwarp();
                        if (valid) {
                            uint4* dst = reinterpret_cast<uint4*>(p.ypool + static_cast<size_t>(row) * p.H + ti.cb * 256 + half * 128 + 32 * q);
#pragma unroll
                            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tempty(as));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int LAYER, int BN>
static cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                              cudaStream_t stream) {
    using C = GemmCfg<BN>;
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<LAYER, BN>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (err != cudaSuccess) return err;
    grouped_gemm_kernel<LAYER, BN><<<a.num_ctas, 192, C::SMEM, stream>>>(tmA, tmB, a);
    return cudaGetLastError();
}

cudaError_t launch_gemm(int layer, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                        cudaStream_t stream) {
    switch (a.tile_n * 10 + layer) {
        case 321: return launch_one<1, 32>(tmA, tmB, a, stream);
        case 322: return launch_one<2, 32>(tmA, tmB, a, stream);
        case 641: return launch_one<1, 64>(tmA, tmB, a, stream);
        case 642: return launch_one<2, 64>(tmA, tmB, a, stream);
        case 961: return launch_one<1, 96>(tmA, tmB, a, stream);
        case 962: return launch_one<2, 96>(tmA, tmB, a, stream);
        case 1281: return launch_one<1, 128>(tmA, tmB, a, stream);
        case 1282: return launch_one<2, 128>(tmA, tmB, a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moeffn
