// Internal launch interface between the C-ABI host code and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moeffn {

struct DevStatus;

// Tile bounds from 48 to 144 rows use the 144-row stage layout, which has a
// paired form: every expert's rows are split into an even number of equal
// token tiles, and the two tiles of a pair share each weight stage of the
// grouped GEMM (two MMA warps, one per tile, consume every stage).  The host
// pairs when an expert is expected to have more than one tile.
constexpr bool pairable_tile_n(int tile_n) { return tile_n > 32 && tile_n <= 144; }

struct LayoutArgs {
    const uint8_t* x;
    const uint32_t* x_sf;
    const int64_t* topk_idx;
    const float* topk_w;
    int T, H, E, k, tile_n;   // tile_n: most token rows per GEMM tile
    int paired;               // an even number of tiles per expert (pairable_tile_n(tile_n) only)
    int* hist;      // [ceil(T*k/1024)][E]
    int* rank;      // [T*k]
    int* counts;    // [E]
    int* offsets;   // [E+1]
    int* tiles;     // [E+1] first token tile of each expert
    int* tile_rows; // [E]   token rows per tile of each expert (multiple of 16)
    int* tile_rec;  // [NT_max][8] per token tile: expert, its first token tile, its token
                    // tiles, rows per tile, its pool offset, its rows, 0, 0
    int* l1_done;   // [NT_max] zeroed here: per token tile, L1 epilogue warps done
    int* slots;     // [T*k]
    int* row2tk;    // [P_max]
    float* wpool;   // [P_max]
    int* slack;     // [P_max/128]
    uint8_t* xpool;       // [P_max][H]
    uint32_t* xpool_sf;   // [NT_max][H/128][2][128]
    DevStatus* status;
    int P_max, NT_max;    // pool rows and token tiles the workspace holds (bounds-checked builds)
};

struct PrepareArgs {
    const uint8_t* w1;
    const uint32_t* w1_sf;
    const uint8_t* w2;
    const uint32_t* w2_sf;
    uint8_t* w1p;
    uint32_t* w1p_sf;
    uint8_t* w2p;
    uint32_t* w2p_sf;
    int H, I, E;
};

// One grouped GEMM launch (L1: Xpool x W1 with the SwiGLU/requant epilogue;
// L2: Hpool x W2 with the BF16 epilogue).
struct GemmArgs {
    const int* tiles;        // [E+1] first token tile of each expert (tiles[E]: all tiles)
    const int* tile_rec;     // per token tile: its expert's tile record (LayoutArgs)
    int E;
    int H, I;
    const float* wpool;
    uint8_t* hpool;         // L1 output [P_max][I]
    uint8_t* hpool_sf;      // L1 output scales (per token tile, per K block of L2)
    uint16_t* ypool;        // L2 output [P_max][H]
    DevStatus* status;
    uint64_t timeout_ns;
    int debug_flags;
    float act_clamp;        // > 0: L1 epilogue clamps gate <= c and -c <= up <= c
    int fast_math;          // 1: SiLU with approximate exp and reciprocal
    int num_sms;
    int tile_n;             // most token rows per tile (selects the stage layout)
    int paired;             // pairs of token tiles per stage (LayoutArgs::paired)
    int run_l1, run_l2;     // which layers' items this launch runs (L1 items first)
    int* l1_done;           // [NT_max] per token tile: L1 epilogue warps that published their rows
};

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int64_t* idx, float* w,
                              cudaStream_t stream);
cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t stream);
cudaError_t launch_combine(const uint16_t* ypool, const int* slots, int T, int H, int k,
                           uint16_t* y, int P_max, DevStatus* status, cudaStream_t stream);
cudaError_t launch_prepare(const PrepareArgs& a, cudaStream_t stream);
// Tensor maps of one grouped GEMM launch: the prepared weights (boxes of
// 128 rows x 128 K), the token pool (boxes of 8, 16, ..., kMaxTileN/2 rows,
// half a pair's tile), and the scale arrays as rows of 512 B (weights: one
// per 128-row block and K block) and of 1 KB (pool: one per token tile and K
// block), read as boxes of one row (512 B or 1 KB of the pool row).
struct GemmMaps {
    CUtensorMap a;
    CUtensorMap b[14];
    CUtensorMap sfa;
    CUtensorMap sfb_512, sfb_1k;
};
// One launch of the grouped GEMM kernel over the L1 items (a.run_l1), then
// the L2 items (a.run_l2): with both, each L2 item waits for the L1 items of
// its token tile (counters a.l1_done); m1 and m2 are the two layers' maps.
cudaError_t launch_gemm(const GemmMaps& m1, const GemmMaps& m2, const GemmArgs& a, cudaStream_t stream);

}  // namespace moeffn
