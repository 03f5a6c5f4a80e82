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
// block, one scale byte selected per MMA; the 2-SM MMA of a CTA pair) and
// 4.6 "Epilogue warps".
//
// GB300 design (not the pages' SM100 kernel):
//  - Clusters of two CTAs on two SMs run a 2-SM MMA (cta_group::2): M = 256
//    weight rows (128 staged and accumulated per CTA) x N token columns (N/2
//    staged per CTA).  Every CTA keeps its own weight-row scales and the
//    full token-tile scales in its tensor memory.  A stage therefore holds
//    one 128-row weight tile and half a token tile per SM.
//  - A block-scaled MMA (K = 32) occupies an SM's tensor core for
//    max(48, N/2) cycles, so token tiles are wide: each expert's rows are
//    split into equal tiles of a multiple of 16 rows, at most 144 (most
//    experts), 224 (more than ~272 rows per expert) or 32 (decode-sized
//    batches, where narrow stages allow 10 in flight).
//  - Persistent: pair p takes work items p, p + P, ...; the even and the odd
//    ones go to two MMA warps, each with its own ring of stages (4 for tiles
//    of at most 144 rows) fed by its own TMA warp; twelve warps drain TMEM.
//    Items use accumulator regions in turn (three of 144 columns, two of
//    224 or four of 32), so an MMA warp rarely waits for the epilogue.
//  - Paired tiles (when experts expect more than one tile): every expert has
//    an even number of tiles, and the two tiles of one weight block share
//    each weight stage of a single ring: per K block the stage holds the
//    weight tile once and both token halves, and MMA warp w issues tile w's
//    MMAs.  The weights then cross L2 and shared memory once per two tiles.
//  - The epilogue loads a finished region's chunks as BF16 pairs (both
//    layers round the accumulators to BF16 first) and frees the region before
//    any arithmetic, so the next item's MMAs start within a few hundred cycles.
//  - The MMA and TMA warps issue from all 32 lanes through elect.sync; the
//    forward's kernels use programmatic dependent launch.
//  - For L1 a CTA's 128 weight rows are gate and up of 64 channels in bands
//    of 32; the warps draining the gate and the up band of a channel group
//    each finish half of a chunk's tokens, exchanging the other half through
//    shared memory, for SwiGLU and requantisation.
//  - Scale factors of a token tile are stored per tile in tensor-memory copy
//    order (two 512-byte chunks per 128-wide K block).
#include "common.cuh"
#include "kernels.h"

#include <cuda_bf16.h>

namespace moeffn {

// warp roles: 0..11 drain TMEM (three warps per lane quarter, taking every
// third 32-column chunk); 12 and 13 issue the MMAs of the even and the odd
// tiles of the pair (leader; idle in the peer); 14 and 15 issue the TMA
// copies of the two rings of stages, or 14 alone those of the one paired
// ring (both CTAs; the copies of both signal the leader's barrier of the
// stage).  The MMA and TMA
// warps issue from all 32 lanes through elect.sync: issued from one lane of a
// divergent branch a block-scaled MMA costs about twice its tensor-pipe time.
constexpr int kEpiWarps = 12;
constexpr int kEpiGroups = kEpiWarps / 4;
constexpr int kMmaWarps = 2;
constexpr int kFirstMmaWarp = kEpiWarps;
constexpr int kFirstProducerWarp = kFirstMmaWarp + kMmaWarps;
constexpr int kMaxProducersPerRing = 1;
// L1 epilogue: the gate and the up warp of a channel group hand each other one
// half of a 32-token chunk through a 32-channel x 16-token BF16 buffer
constexpr int kXchLd = 18;                           // BF16 per buffer row: 16 tokens + 2 padding
constexpr int kXchElems = 32 * kXchLd;

// producer warps of a ring of `sr` stages: the largest divisor of sr up to kMaxProducersPerRing
constexpr int pick_producers(int sr) {
    int best = 1;
    for (int p = 1; p <= kMaxProducersPerRing; ++p)
        if (sr % p == 0) best = p;
    return best;
}

// BN: widest token tile of the stage layout; RW: TMEM columns of one
// accumulator region (the widest tile it holds).  NACC regions are used in
// turn by the tiles of a pair (tile i -> region i % NACC), so with three or
// more regions an MMA warp starts its next tile while the epilogue still
// drains its previous one.  PAIRED: one ring whose stages hold one weight
// tile and the halves of two token tiles of its expert (MMA warp w takes
// token tile w of every stage); otherwise one ring per MMA warp, one token
// tile per stage.
template <int BN, int RW, bool PAIRED>
struct GemmCfg {
    static constexpr int TPS = PAIRED ? 2 : 1;          // token tiles per stage
    static constexpr int BH = BN / 2;                   // token rows staged per CTA and tile, at most
    static constexpr int A_BYTES = 128 * 128;           // 128 weight rows x 128 K (E2M1, 16-byte padded)
    // a TMA load of packed E2M1 (16U4_ALIGN16B) signals the packed global bytes
    // as its transaction count although it fills A_BYTES of shared memory
    static constexpr int A_TX_BYTES = A_BYTES / 2;
    static constexpr int B_BYTES = BH * 128;            // a multiple of 1024 (BH: a multiple of 8)
    // operand tiles of a stage, 1024-byte aligned for the 128-byte swizzle
    static constexpr int STAGE_BYTES = (A_BYTES + TPS * B_BYTES + 1023) / 1024 * 1024;
    // scales of a stage, kept apart from the tiles: 512 B weight-row scales,
    // then per token tile one 512-byte chunk of token scales per 128 tile rows
    static constexpr int SFB_BYTES = BN <= 128 ? 512 : 1024;
    static constexpr int SF_STAGE = 512 + TPS * SFB_BYTES;
    // per gate/up warp pair two BF16 exchange buffers (L1); per pair warp a vote word
    static constexpr int XCH_BYTES = (kEpiWarps / 2) * 2 * kXchElems * 2;
    static constexpr int EPI_BYTES = XCH_BYTES + 4 * kEpiWarps;
    static constexpr int FIXED = 1024 + EPI_BYTES + 256;
    static constexpr int STAGES_FIT = (232448 - FIXED) / (STAGE_BYTES + SF_STAGE);
    static constexpr int STAGES_CAP = STAGES_FIT > 12 ? 12 : STAGES_FIT;
    static constexpr int RINGS = PAIRED ? 1 : kMmaWarps;
    static constexpr int RING = STAGES_CAP / RINGS;            // stages per ring
    static constexpr int STAGES = RINGS * RING;
    static constexpr int PRODUCERS = pick_producers(RING);     // producer warps per ring
    static constexpr int THREADS = 32 * (kEpiWarps + kMmaWarps + RINGS * PRODUCERS);
    static constexpr int SMEM = FIXED + STAGES * (STAGE_BYTES + SF_STAGE);
    static constexpr int SF_SET_COLS = 12;              // SFA 4 | SFB 8; per MMA warp two sets alternating by K block
    static constexpr int SF_COLS = kMmaWarps * 2 * SF_SET_COLS;
    static constexpr int NACC_FIT = (512 - SF_COLS) / RW;
    static constexpr int NACC = NACC_FIT > 4 ? 4 : NACC_FIT;   // accumulator regions
    static constexpr int SF_COL = NACC * RW;
    static constexpr int TMEM_NEED = NACC * RW + SF_COLS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
    // 32-column chunks of a region per epilogue warp, at most
    static constexpr int MAXC = ((RW + 31) / 32 + kEpiGroups - 1) / kEpiGroups;
    static_assert(TMEM_NEED <= 512, "tensor memory overflow");
    static_assert(BN % 16 == 0 && BN <= kMaxTileN && RW % kTileQuantum == 0 && RW <= BN, "token tile");
    static_assert(SMEM <= 232448, "shared memory");
    static_assert(NACC >= 2, "at least two accumulator regions");
    static_assert(RING >= 2, "pipeline too shallow");
    static_assert(RING % PRODUCERS == 0, "each producer warp owns whole stages");
    static_assert(B_BYTES % 1024 == 0, "second token tile of a stage on a swizzle-atom boundary");
};

// token-tile TMA boxes per CTA (half a tile): 8, 16, ..., kMaxTileN / 2 rows
struct TokenMaps {
    CUtensorMap m[kNumTokenBoxes];
};
__device__ __forceinline__ int box_for_half(int n) {
    return n <= 8 ? 0 : (n + 7) / 8 - 1;
}
__device__ __forceinline__ int box_half_rows(int box) {
    return 8 * (box + 1);
}

static_assert(sizeof(GemmMaps::b) / sizeof(CUtensorMap) == kNumTokenBoxes, "one token map per box height");

struct TileInfo {
    int e, cb, tile_idx, row0, nvalid, ncols;   // ncols: pair MMA N (the expert's tile rows, a multiple of 16)
};

// Work items run expert by expert; within an expert, weight-row tile by tile
// and, inside one, token tile by token tile.  Expert e owns items
// [tiles[e] * ncb, tiles[e + 1] * ncb), so item t / ncb is one of e's token
// tiles, whose 32-byte record holds what decoding item t needs.  The loops
// load the next item's record while they work on the current item.
struct TileRec {
    int4 a;   // expert, its first token tile, its token tiles, rows per tile
    int4 b;   // its first pool row, its rows
};
__device__ __forceinline__ TileRec load_rec(int t, int ncb, const GemmArgs& p) {
    const int4* r = reinterpret_cast<const int4*>(p.tile_rec) + 2 * (t / ncb);
    return TileRec{__ldg(r), __ldg(r + 1)};
}
__device__ __forceinline__ TileInfo decode_rec(int t, int ncb, const TileRec& r) {
    TileInfo ti;
    const int t0 = r.a.y, ntb = r.a.z, rows = r.a.w;
    const int local = t - t0 * ncb;
    ti.e = r.a.x;
    ti.cb = local / ntb;
    const int nb = local - ti.cb * ntb;
    ti.tile_idx = t0 + nb;
    ti.row0 = r.b.x + nb * rows;
    ti.nvalid = min(rows, r.b.y - nb * rows);
    ti.ncols = rows;
    return ti;
}

// The tensor maps of one layer (kernel parameters).
struct LayerMaps {
    CUtensorMap a;      // prepared weights, boxes of 128 rows x 128 K
    CUtensorMap sfa;    // weight scales, one 512-B row per box
    CUtensorMap sfb;    // pool scales, one row (512 B or 1 KB) per box
    TokenMaps b;        // token pool, boxes of 8 .. kMaxTileN / 2 rows
};

// The items of one launch: n1 L1 items (indices [0, n1)) then n2 L2 items.
// Within a layer, item u covers token tile u / ncb and weight block u % ncb
// of that tile's expert (see decode_rec).
struct Sched {
    int n1, n;                 // L1 items, all items
    int ncb1, ncb2;            // 256-row weight blocks per expert (W1: 2I rows, W2: H rows)
    int nkb1, nkb2;            // 128-wide K blocks (L1: H, L2: I)
    int rows1, rows2;          // weight rows per expert
    __device__ __forceinline__ int ncb(int layer) const { return layer == 1 ? ncb1 : ncb2; }
    __device__ __forceinline__ int nkb(int layer) const { return layer == 1 ? nkb1 : nkb2; }
    __device__ __forceinline__ int rows(int layer) const { return layer == 1 ? rows1 : rows2; }
};
__device__ __forceinline__ int item_layer(int t, const Sched& s) { return t < s.n1 ? 1 : 2; }
__device__ __forceinline__ int item_local(int t, const Sched& s) { return t < s.n1 ? t : t - s.n1; }
__device__ __forceinline__ TileRec item_rec(int t, const Sched& s, const GemmArgs& p) {
    return load_rec(item_local(t, s), s.ncb(item_layer(t, s)), p);
}
__device__ __forceinline__ TileInfo item_info(int t, const Sched& s, const TileRec& r) {
    return decode_rec(item_local(t, s), s.ncb(item_layer(t, s)), r);
}

// Wait, bounded, until every L1 item of a token tile has published its rows:
// one lane polls the tile's counter with acquire loads at GPU scope; on
// success the warp orders its later asynchronous-proxy reads (TMA loads of
// those rows) after the rows the counter published.
__device__ __forceinline__ bool wait_l1_rows(const int* ctr, int target, volatile int* abort, uint64_t timeout_ns,
                                             DevStatus* st) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v < target) {
            const uint64_t t0 = global_timer_ns();
            while (true) {
                __nanosleep(64);
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
                if (v >= target) break;
                if (*abort) { ok = 0; break; }
                if (global_timer_ns() - t0 > timeout_ns) {
                    atomicOr(&st->code, DEV_ERR_TIMEOUT);
                    atomicCAS(&st->detail, 0u, 7u);
                    *abort = 1;
                    ok = 0;
                    break;
                }
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) asm volatile("fence.proxy.async.global;" ::: "memory");
    return ok != 0;
}

// the 64 threads of gate/up warp pair pi = 2 * group + pair (warps 2 pi, 2 pi + 1)
__device__ __forceinline__ void pair_sync(int pi) {
    switch (pi) {
        case 0: named_barrier_sync<1>(64); break;
        case 1: named_barrier_sync<2>(64); break;
        case 2: named_barrier_sync<3>(64); break;
        case 3: named_barrier_sync<4>(64); break;
        case 4: named_barrier_sync<5>(64); break;
        default: named_barrier_sync<6>(64); break;
    }
}

template <int BN, int RW, bool PAIRED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GemmCfg<BN, RW, PAIRED>::THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ LayerMaps m1, const __grid_constant__ LayerMaps m2,
                    const GemmArgs p) {
    using C = GemmCfg<BN, RW, PAIRED>;
    constexpr int S = C::STAGES, ACC = C::NACC;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);
    const uint32_t sfbase = sbase + S * C::STAGE_BYTES;                  // [S][SF_STAGE] scales
    uint8_t* epi_base = gbase + S * (C::STAGE_BYTES + C::SF_STAGE);
    __nv_bfloat16* xch = reinterpret_cast<__nv_bfloat16*>(epi_base);    // [6 pairs][2][32][kXchLd]
    volatile int* pair_ok = reinterpret_cast<volatile int*>(epi_base + C::XCH_BYTES);   // [6 pairs][2 warps]
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi_base + C::EPI_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (S + s); };
    auto tfull = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto tempty = [&](int a) { return bar0 + 8u * (2 * S + ACC + a); };
    const uint32_t mma_done = bar0 + 8u * (2 * S + 2 * ACC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2 * ACC + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_cta_rank();           // 0: leader (issues the MMAs), 1: peer
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // the leader's "stage full" counts the bytes of both CTAs' copies
            // (they signal it directly); the peer's own is unused.  A paired
            // stage is free once both MMA warps' reads of it are complete.
            mbar_init(full(s), 1);
            mbar_init(empty(s), PAIRED ? kMmaWarps : 1);
        }
        for (int a = 0; a < ACC; ++a) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), 2 * kEpiWarps);         // one arrival per epilogue warp of both CTAs
        }
        mbar_init(mma_done, kMmaWarps);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&m1.a);
        prefetch_tensormap(&m1.sfa);
        prefetch_tensormap(&m1.sfb);
        prefetch_tensormap(&m2.a);
        prefetch_tensormap(&m2.sfa);
        prefetch_tensormap(&m2.sfb);
    }
    if (warp == kFirstMmaWarp) {
        tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                                      // both CTAs' barriers exist before any copy signals one
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();                                          // the previous kernel's tables and pools are written
    pdl_launch_dependents();

    const int npairs = gridDim.x >> 1, pair = blockIdx.x >> 1;
    Sched sc;
    sc.ncb1 = p.I / 128;
    sc.ncb2 = (p.H + 255) / 256;
    sc.nkb1 = p.H / 128;
    sc.nkb2 = p.I / 128;
    sc.rows1 = 2 * p.I;
    sc.rows2 = p.H;
    {
        const int tiles = __ldg(p.tiles + p.E);
        sc.n1 = p.run_l1 ? tiles * sc.ncb1 : 0;
        sc.n = sc.n1 + (p.run_l2 ? tiles * sc.ncb2 : 0);
    }
    const int total = sc.n;
    // an L2 item in the same launch as the L1 items waits for its token tile's rows
    const bool wait_l1 = sc.n1 > 0;
    const int l1_target = 2 * kEpiWarps * sc.ncb1;    // one count per epilogue warp of both CTAs per L1 item
    // Items of this pair in the order its MMA warps and its epilogue take them.
    // Paired: items 2u and 2u + 1 (the two token tiles of one weight block,
    // every expert having an even number of tiles) form unit u, units u = pair,
    // pair + P, ... run in turn, MMA warp w taking item 2u + w.  Otherwise MMA
    // warp w takes items pair + w P, pair + (w + 2) P, ...  Either way the
    // pair's i-th item has ordinal i and accumulator region i % NACC.
    auto item_at = [&](int i) {
        return PAIRED ? 2 * (pair + (i >> 1) * npairs) + (i & 1) : pair + i * npairs;
    };

    if (warp >= kFirstProducerWarp) {
        // ------------------------------------------------------------ TMA (both CTAs)
        const int ring = (warp - kFirstProducerWarp) / C::PRODUCERS;
        const int pw = (warp - kFirstProducerWarp) % C::PRODUCERS;
        {
            // the whole warp runs the loop; one elected lane issues each copy.
            // Both CTAs' copies of a stage signal the leader's "stage full",
            // which the leader arms with the bytes of both halves.
            const uint32_t leader_full0 = map_shared_rank(full(0), 0);
            int ls = 0;                                  // stage within the ring
            uint32_t phase = 0;
            uint32_t armed[C::RING] = {};
            const bool starve = (p.debug_flags & 1) && rank == 0 && ring == 0;
            bool ok = true;
            // item sequence of this ring: paired, the first item of every unit
            const int t_first = PAIRED ? item_at(0) : pair + ring * npairs;
            const int t_step = 2 * npairs;
            TileRec rec = t_first < total ? item_rec(t_first, sc, p) : TileRec{};
            for (int t = t_first; t < total && ok; t += t_step) {
                const TileInfo ti = item_info(t, sc, rec);
                const int layer = item_layer(t, sc);
                const LayerMaps& m = layer == 1 ? m1 : m2;
                const int nkb = sc.nkb(layer), a_rows = sc.rows(layer);
                if (t + t_step < total) rec = item_rec(t + t_step, sc, p);
                if (layer == 2 && wait_l1) {
                    bool rows_ok = wait_l1_rows(p.l1_done + ti.tile_idx, l1_target, abort_flag, p.timeout_ns,
                                                p.status);
                    if (PAIRED && rows_ok)
                        rows_ok = wait_l1_rows(p.l1_done + ti.tile_idx + 1, l1_target, abort_flag, p.timeout_ns,
                                               p.status);
                    if (!rows_ok) {
                        ok = false;
                        break;
                    }
                }
                const int mrow = ti.cb * 256 + 128 * static_cast<int>(rank);   // first weight row of this CTA
                const bool mine_valid = mrow < a_rows;                          // false only for an L2 tail half
                const int a0 = ti.e * a_rows + mrow;
                const int sf_block = (ti.e * a_rows + (mine_valid ? mrow : ti.cb * 256)) / 128;
                const int sfa_row = sf_block * nkb;          // rows of 512 B: one per 128-row block and K block
                const int sfb_row = ti.tile_idx * nkb;       // rows of 1 KB: one per token tile and K block
                const int half = ti.ncols / 2;
                const int box = box_for_half(half);
                const CUtensorMap* tmBox = &m.b.m[box];
                const int brow = ti.row0 + half * static_cast<int>(rank);
                // paired: the unit's second tile is the next tile of the expert
                // (rows ti.ncols further on, scale rows nkb further on)
                const uint32_t bytes =
                    C::A_TX_BYTES + C::TPS * (box_half_rows(box) * 128 + C::SFB_BYTES) + 512;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (ls % C::PRODUCERS != pw) {
                        if (++ls == C::RING) {
                            ls = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    const int stage = ring * C::RING + ls;
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag,
                                                                    p.timeout_ns, p.status, 1))) {
                        ok = false;
                        break;
                    }
                    const uint32_t sb = sbase + stage * C::STAGE_BYTES;
                    const uint32_t ss = sfbase + stage * C::SF_STAGE;
                    if (!(starve && t == t_first && layer == 1 && kb == 0)) {
                        const uint32_t fb = leader_full0 + 8u * stage;
                        if (rank == 0) mbar_arrive_expect_tx_w(full(stage), 2 * bytes);
                        tma_load_2d_pair_w(sb, &m.a, fb, kb * 128, a0);
                        tma_load_2d_pair_w(sb + C::A_BYTES, tmBox, fb, kb * 128, brow);
                        tma_load_2d_pair_w(ss, &m.sfa, fb, 0, sfa_row + kb);
                        tma_load_2d_pair_w(ss + 512, &m.sfb, fb, 0, sfb_row + kb);
                        if (PAIRED) {
                            tma_load_2d_pair_w(sb + C::A_BYTES + C::B_BYTES, tmBox, fb, kb * 128, brow + ti.ncols);
                            tma_load_2d_pair_w(ss + 512 + C::SFB_BYTES, &m.sfb, fb, 0, sfb_row + nkb + kb);
                        }
                        ++armed[ls];
                    }
                    if (++ls == C::RING) {
                        ls = 0;
                        phase ^= 1u;
                    }
                }
            }
            // never leave copies in flight into shared memory: the leader waits
            // for the last arming of every stage of its ring to land (immediate
            // on the normal path; it counts the peer's bytes too).  The peer's
            // copies are consumed by the leader's MMAs before the pair's final
            // cluster barrier; after a timeout the peer leaves its loop only once
            // its own bounded wait for a free stage ran out, long after its last
            // copies landed.
            if (rank == 0)
                for (int l = 0; l < C::RING; ++l)
                    if (armed[l])
                        mbar_wait_bounded(full(ring * C::RING + l), (armed[l] - 1u) & 1u, abort_flag,
                                          p.timeout_ns, p.status, 5, false);
        }
        __syncwarp();
    } else if (warp >= kFirstMmaWarp) {
        const int mw = warp - kFirstMmaWarp;                 // this warp's items (see item_at)
        if (rank == 0) {
            // ---------------------------------------------------- MMA (leader)
            // the whole warp runs the loop; one elected lane issues each instruction
            constexpr uint32_t IDESC = idesc_mx_e2m1_e4m3(256, 0);
            int ls = 0, it = 0;
            uint32_t phase = 0, kiter = 0;
            bool ok = true;
            const uint32_t sf_base = tmem + C::SF_COL + static_cast<uint32_t>(mw * 2 * C::SF_SET_COLS);
            // paired: this warp's token tile of every stage of the one ring
            const int ring = PAIRED ? 0 : mw;
            const uint32_t b_off = C::A_BYTES + (PAIRED ? mw * C::B_BYTES : 0);
            const uint32_t sfb_off = 512 + (PAIRED ? mw * C::SFB_BYTES : 0);
            const int t_first = PAIRED ? 2 * pair + mw : pair + mw * npairs;
            TileRec rec = t_first < total ? item_rec(t_first, sc, p) : TileRec{};
            for (int t = t_first; t < total && ok; t += 2 * npairs, ++it) {
                const TileInfo ti = item_info(t, sc, rec);
                const int nkb = sc.nkb(item_layer(t, sc));
                if (t + 2 * npairs < total) rec = item_rec(t + 2 * npairs, sc, p);
                const uint32_t idesc_n = IDESC | (static_cast<uint32_t>(ti.ncols >> 3) << 17);
                const bool two_sfb = ti.ncols > 128;
                const int tord = 2 * it + mw;                  // ordinal of this tile in the pair's sequence
                const int as = tord % ACC;
                const uint32_t ap = static_cast<uint32_t>(tord / ACC) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded<true>(tempty(as), ap ^ 1u, abort_flag, p.timeout_ns,
                                                                     p.status, 2)))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(as * RW);
                uint32_t idk[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    idk[k] = idesc_n | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
                for (int kb = 0; kb < nkb; ++kb) {
                    const int stage = ring * C::RING + ls;
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(full(stage), phase, abort_flag, p.timeout_ns,
                                                                    p.status, 3))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sb = sbase + stage * C::STAGE_BYTES;
                    const uint32_t ss = sfbase + stage * C::SF_STAGE;
                    const uint32_t sfs = sf_base + (kiter & 1u) * C::SF_SET_COLS;
                    ++kiter;
                    // descriptors of the stage; a K step of 32 bytes adds 2 to the address field
                    const uint64_t adesc = desc_kmajor_sw128(sb), bdesc = desc_kmajor_sw128(sb + b_off);
                    tc_cp_sf_pair_w(sfs, desc_sf_block(ss));
                    tc_cp_sf_pair_w(sfs + 4, desc_sf_block(ss + sfb_off));
                    if (two_sfb) tc_cp_sf_pair_w(sfs + 8, desc_sf_block(ss + sfb_off + 512));
                    tc_mma_mx_pair_w(d, adesc, bdesc, idk[0], sfs, sfs + 4, kb != 0);
                    tc_mma_mx_pair_w(d, adesc + 2, bdesc + 2, idk[1], sfs, sfs + 4, 1u);
                    tc_mma_mx_pair_w(d, adesc + 4, bdesc + 4, idk[2], sfs, sfs + 4, 1u);
                    tc_mma_mx_pair_w(d, adesc + 6, bdesc + 6, idk[3], sfs, sfs + 4, 1u);
                    tc_commit_pair_w(empty(stage));
                    if (++ls == C::RING) {
                        ls = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit_pair_w(tfull(as));
            }
            // every MMA issued by the MMA warps is complete before TMEM is freed
            // (a kernel uses either 1-CTA or 2-CTA tcgen05 forms, never both)
            tc_commit_pair_w(mma_done);
            mbar_wait_bounded(mma_done, 0, abort_flag, p.timeout_ns, p.status, 6, false);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;                              // TMEM lane quarter of this warp
        const int grp = warp >> 2;                           // this warp takes chunks grp, grp + 3, ...
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
        const uint32_t leader_tempty0 = map_shared_rank(tempty(0), 0);
        TileRec rec = item_at(0) < total ? item_rec(item_at(0), sc, p) : TileRec{};
        for (int it = 0;; ++it) {
            const int t = item_at(it);
            if (t >= total) break;
            const TileInfo ti = item_info(t, sc, rec);
            const bool l1 = item_layer(t, sc) == 1;
            if (item_at(it + 1) < total) rec = item_rec(item_at(it + 1), sc, p);
            const int as = it % ACC;
            const uint32_t ap = static_cast<uint32_t>(it / ACC) & 1u;
            const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(tfull(as), ap, abort_flag, p.timeout_ns,
                                                                        p.status, 4));
            if (l1) {
                // the two warps of a gate/up pair meet at named barriers below, so
                // they decide together whether to go on (a timeout may reach only one)
                const int pi = warp >> 1, hs = q & 1;
                if (lane == 0) pair_ok[pi * 2 + hs] = got ? 1 : 0;
                pair_sync(pi);
                const bool both = pair_ok[pi * 2] && pair_ok[pi * 2 + 1];
                pair_sync(pi);
                if (!both) break;
            } else if (!got) {
                break;
            }
            tc_fence_after();
            const uint32_t tacc = tq + static_cast<uint32_t>(as * RW);
            const int nchunks = (ti.nvalid + 31) / 32;
            const int mrow = ti.cb * 256 + 128 * static_cast<int>(rank);
            // L1: quarter q holds band q of this CTA's 128 rows: gate (q even) or
            // up (q odd) of channels cbase1 + [0, 32), cbase1 = mrow / 2 + 32 (q / 2);
            // thread `lane` has channel cbase1 + lane for the chunk's 32 tokens
            const int hs = q & 1;
            const int cbase1 = mrow / 2 + 32 * (q >> 1);
            // This warp's chunks (grp + 3 c) of the region, as BF16 pairs: pk[c][i]
            // holds tokens 2 i and 2 i + 1.  Both epilogues round the accumulators to
            // BF16 first, so the region is released before any arithmetic on them.
            uint32_t pk[C::MAXC][16];
#pragma unroll
            for (int c = 0; c < C::MAXC; ++c) {
                const int j = grp + kEpiGroups * c;
                if (j < nchunks) {
                    uint32_t r[32];
                    tmem_ld32_issue(tacc + 32 * j, r);
                    tmem_ld_wait(r);
                    if (l1 && (p.debug_flags & 2)) {
                        // test hook: raw FP32 accumulators, [P_max][gate I | up I] floats
                        float* zd = reinterpret_cast<float*>(p.ypool);
#pragma unroll
                        for (int n = 0; n < 32; ++n)
                            if (32 * j + n < ti.nvalid)
                                zd[static_cast<size_t>(ti.row0 + 32 * j + n) * 2 * p.I + hs * p.I + cbase1 + lane] =
                                    __uint_as_float(r[n]);
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) pk[c][i] = bf16x2_bits(r[2 * i], r[2 * i + 1]);
                }
            }
            tc_fence_before();
            __syncwarp();
            // relaxed: what the MMA warp must not overtake are this warp's TMEM loads,
            // complete (tcgen05.wait::ld) and fenced above; the rows stored to global
            // memory are not read by that warp, and a release would wait for them
            if (lane == 0) mbar_arrive_remote_relaxed(leader_tempty0 + 8u * as);
            if (l1) {
                // The gate warp finishes tokens 0-15 of a chunk and the up warp tokens
                // 16-31; each hands the other the half of its values that it needs.
                const int pi = warp >> 1;
                __nv_bfloat16* XG = xch + (2 * pi) * kXchElems;     // gate of tokens 16-31, for the up warp
                __nv_bfloat16* XU = XG + kXchElems;                 // up of tokens 0-15, for the gate warp
                const int cbase = cbase1;
                const int mine0 = 16 * hs;                          // first token of this warp's half
                const float clamp = p.act_clamp;
#pragma unroll
                for (int c = 0; c < C::MAXC; ++c) {
                    const int j = grp + kEpiGroups * c;
                    if (j >= nchunks) break;                        // the same for both warps of the pair
                    // this warp's half and the half it hands over (constant indices, so
                    // that pk stays in registers)
                    uint32_t mw2[8], ow2[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        mw2[i] = hs ? pk[c][8 + i] : pk[c][i];
                        ow2[i] = hs ? pk[c][i] : pk[c][8 + i];
                    }
                    __nv_bfloat16* give = hs ? XU : XG;
#pragma unroll
                    for (int i = 0; i < 8; ++i) *reinterpret_cast<uint32_t*>(give + lane * kXchLd + 2 * i) = ow2[i];
                    // top-k weights of this half's 16 tokens, one per lane, broadcast below
                    const int r16 = 32 * j + mine0 + (lane & 15);
                    const float wl = r16 < ti.nvalid ? __ldg(p.wpool + ti.row0 + r16) : 0.f;
                    pair_sync(pi);
                    const __nv_bfloat16* take = hs ? XG : XU;
                    float g[16], u[16];
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const float2 o = __bfloat1622float2(
                            *reinterpret_cast<const __nv_bfloat162*>(take + lane * kXchLd + i));
                        const float m0 = bf16_lo(mw2[i / 2]), m1 = bf16_hi(mw2[i / 2]);
                        g[i] = hs ? o.x : m0;
                        u[i] = hs ? m0 : o.x;
                        g[i + 1] = hs ? o.y : m1;
                        u[i + 1] = hs ? m1 : o.y;
                    }
                    if (clamp > 0.f) {
                        // optional activation clamp (MegaMoE notes, "Activation clamp"):
                        // the gate from above only, the up projection on both sides
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            g[i] = fminf(g[i], clamp);
                            u[i] = fminf(fmaxf(u[i], -clamp), clamp);
                        }
                    }
                    float h[16];
                    if (p.fast_math) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) h[i] = silu_fast(g[i]) * u[i] * __shfl_sync(0xffffffffu, wl, i);
                    } else {
                        // two tokens at a time in packed FP32x2 arithmetic: the same roundings,
                        // (silu(g) * u) * w, as the scalar form
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const float2 s = silu_x2(make_float2(g[i], g[i + 1]));
                            const float2 wt = make_float2(__shfl_sync(0xffffffffu, wl, i), __shfl_sync(0xffffffffu, wl, i + 1));
                            const float2 hv = __fmul2_rn(__fmul2_rn(s, make_float2(u[i], u[i + 1])), wt);
                            h[i] = hv.x;
                            h[i + 1] = hv.y;
                        }
                    }
                    // Per token: amax over the 32 channels of the group (the warp's lanes).
                    // A halving exchange: after the shuffle across lane bit b, a lane keeps
                    // the maxima of half of its tokens, so 8 + 4 + 2 + 1 + 1 shuffles leave
                    // lanes 2 i and 2 i + 1 with the amax of token i.
                    float m8[8], m4[4], m2[2];
                    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float lo = fabsf(h[k]), hi = fabsf(h[k + 8]);
                        m8[k] = fmaxf(b4 ? hi : lo, __shfl_xor_sync(0xffffffffu, b4 ? lo : hi, 16));
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        m4[k] = fmaxf(b3 ? m8[k + 4] : m8[k], __shfl_xor_sync(0xffffffffu, b3 ? m8[k] : m8[k + 4], 8));
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        m2[k] = fmaxf(b2 ? m4[k + 2] : m4[k], __shfl_xor_sync(0xffffffffu, b2 ? m4[k] : m4[k + 2], 4));
                    float m1 = fmaxf(b1 ? m2[1] : m2[0], __shfl_xor_sync(0xffffffffu, b1 ? m2[0] : m2[1], 2));
                    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
                    const int my_ex = requant_exponent(m1);        // of token lane / 2
                    const float my_s = exp2_neg(my_ex);
                    // codes of channel `lane` for this half's 16 tokens, staged as
                    // [token][32 channels] so that each lane then stores 16 bytes of a
                    // row; the staging reuses the hand-over buffer this warp has read
                    // (its partner writes it again only after the next pair barrier)
                    __syncwarp();
                    uint8_t* stg = reinterpret_cast<uint8_t*>(const_cast<__nv_bfloat16*>(take));
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const float2 sv = __fmul2_rn(make_float2(h[i], h[i + 1]),
                                                     make_float2(__shfl_sync(0xffffffffu, my_s, 2 * i),
                                                                 __shfl_sync(0xffffffffu, my_s, 2 * i + 2)));
                        const uint32_t c2 = e4m3x2(sv.x, sv.y);
                        stg[i * 32 + lane] = static_cast<uint8_t>(c2);
                        stg[(i + 1) * 32 + lane] = static_cast<uint8_t>(c2 >> 8);
                    }
                    __syncwarp();
                    // lane: token mine0 + lane / 2, channels cbase + 16 (lane & 1) + [0, 16)
                    const int rc = 32 * j + mine0 + (lane >> 1);
                    const uint4 cv = *reinterpret_cast<const uint4*>(stg + lane * 16);
                    if (rc < ti.nvalid)
                        *reinterpret_cast<uint4*>(p.hpool + static_cast<size_t>(ti.row0 + rc) * p.I + cbase +
                                                  16 * (lane & 1)) = cv;
                    // the L2 B-operand scale of this token and this 32-channel group
                    if ((lane & 1) == 0 && rc < ti.nvalid) {
                        const int kb2 = cbase / 128, byte = (cbase % 128) / 32;
                        const size_t wd = ((static_cast<size_t>(ti.tile_idx) * (p.I / 128) + kb2) * 2 + (rc >> 7)) * 128 +
                                          (rc & 31) * 4 + ((rc & 127) >> 5);
                        p.hpool_sf[wd * 4 + byte] = static_cast<uint8_t>(my_ex + 127);
                    }
                    __syncwarp();                                   // the staging is reused by the next chunk
                    pair_sync(pi);                                  // the buffers are free for the next chunk
                }
            } else if (mrow < p.H) {
                // thread `lane` has output channel cbase + lane for the chunk's 32 tokens.
                // Lanes 2m and 2m + 1 swap halves: the even lane then holds channels
                // (2m, 2m + 1) of tokens 0-15, the odd lane of tokens 16-31, and each
                // stores one BF16 pair per token (the warp writes 64 contiguous bytes)
                const int cbase = mrow + 32 * q;
                const bool odd = lane & 1;
                const int c2 = cbase + (lane & ~1);
#pragma unroll
                for (int c = 0; c < C::MAXC; ++c) {
                    const int j = grp + kEpiGroups * c;
                    if (j >= nchunks) break;
                    const int nrows = min(32, ti.nvalid - 32 * j) - (odd ? 16 : 0);
                    uint16_t* dst = p.ypool + static_cast<size_t>(ti.row0 + 32 * j + (odd ? 16 : 0)) * p.H + c2;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        // tokens 2i, 2i + 1 of this lane's half: the even lane sends its
                        // tokens 16 + 2i, 16 + 2i + 1, the odd lane its tokens 2i, 2i + 1
                        const uint32_t send = odd ? pk[c][i] : pk[c][8 + i];
                        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
                        const uint32_t keep = odd ? pk[c][8 + i] : pk[c][i];
                        const uint32_t ch0 = odd ? recv : keep, ch1 = odd ? keep : recv;   // channels c2, c2 + 1
                        if (2 * i < nrows)
                            *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(2 * i) * p.H) =
                                __byte_perm(ch0, ch1, 0x5410);
                        if (2 * i + 1 < nrows)
                            *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(2 * i + 1) * p.H) =
                                __byte_perm(ch0, ch1, 0x7632);
                    }
                }
            }
            if (l1 && wait_l1) {
                // publish this warp's share of the token tile's L1 rows and scales to
                // the L2 items of the same launch, which read them by TMA (the
                // asynchronous proxy): proxy fence, GPU-scope fence, then one count
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(p.l1_done + ti.tile_idx, 1);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();                                      // no CTA leaves while its pair may still use its memory
    if (warp == kFirstMmaWarp) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::TMEM_COLS);
    }
}

template <int BN, int RW, bool PAIRED>
static cudaError_t launch_one(const GemmMaps& g1, const GemmMaps& g2, const GemmArgs& a, cudaStream_t stream) {
    using C = GemmCfg<BN, RW, PAIRED>;
    auto kernel = grouped_gemm_kernel<BN, RW, PAIRED>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (err != cudaSuccess) return err;
    // persistent grid: as many CTA pairs as can be resident at once (an L2 item
    // waits for L1 items of other pairs, so all pairs must be resident together)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (a.num_sms / 2), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see launch_pdl
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 1) {
        (void)cudaGetLastError();
        clusters = a.num_sms / 2;
    }
    cfg.gridDim = dim3(2 * (clusters < a.num_sms / 2 ? clusters : a.num_sms / 2), 1, 1);
    LayerMaps m1, m2;
    const GemmMaps* g[2] = {&g1, &g2};
    LayerMaps* m[2] = {&m1, &m2};
    for (int l = 0; l < 2; ++l) {
        m[l]->a = g[l]->a;
        m[l]->sfa = g[l]->sfa;
        m[l]->sfb = BN <= 128 ? g[l]->sfb_512 : g[l]->sfb_1k;
        for (int i = 0; i < kNumTokenBoxes; ++i) m[l]->b.m[i] = g[l]->b[i];
    }
    err = cudaLaunchKernelEx(&cfg, kernel, m1, m2, a);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmMaps& m1, const GemmMaps& m2, const GemmArgs& a, cudaStream_t stream) {
    // stage layouts: tiles of at most 32 rows (10 stages in flight, four
    // accumulator regions); tiles of at most 144 rows, one per stage (8 stages,
    // three regions) or paired (5 stages of one weight tile and two token
    // tiles, three regions); tiles of at most kMaxTileN rows (6 stages, two
    // regions)
    static_assert(!pairable_tile_n(32) && pairable_tile_n(48) && pairable_tile_n(144) && !pairable_tile_n(160),
                  "the paired layout is the 144-row one");
    if (a.tile_n <= 32) return launch_one<32, 32, false>(m1, m2, a, stream);
    if (a.tile_n <= 144)
        return a.paired ? launch_one<144, 144, true>(m1, m2, a, stream) : launch_one<144, 144, false>(m1, m2, a, stream);
    return launch_one<kMaxTileN, kMaxTileN, false>(m1, m2, a, stream);
}

}  // namespace moeffn
