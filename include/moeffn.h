/*
 * moeffn.h -- C ABI of the fused MoE expert forward for one GB300 (sm_103a).
 *
 * The calls follow the problem statement of DeepGEMM's MegaMoE as the pages
 * describe it (MegaMoE code-reading notes, "Host wrapper: how to call
 * MegaMoE" and "Out-of-kernel preparation"): FP8 E4M3 tokens x with packed
 * UE8M0 scales x_sf, topk_idx, topk_weights, and two expert weight sets in
 * FP4 E2M1 with packed UE8M0 scales, producing BF16 y.  The one-GPU path is:
 *
 *   moeffn_route_topk      top-k routing from router logits
 *   moeffn_forward         per-expert count -> 128-row padded prefix ->
 *                          (token, k) -> slot table -> gather into the
 *                          expert-sorted pool -> L1 grouped GEMM (E4M3 x E2M1,
 *                          UE8M0 per 32) + SwiGLU x top-k weight + amax ->
 *                          UE8M0 -> E4M3 -> L2 grouped GEMM -> BF16 ->
 *                          top-k combine back to token order
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller (e.g. from
 *    PyTorch); the library allocates and frees nothing.  Host-only calls are
 *    marked as such.
 *  - Row-major, densely packed; element type and shape in each comment.
 *  - E2M1 packing: two codes per byte, element 2i in the low nibble.
 *  - UE8M0 packing: four codes per uint32 along K; byte b (little-endian) of
 *    word w covers K range [128w + 32b, 128w + 32b + 32).  One scale per row
 *    per 32 consecutive K elements (recipe (1, 1, 32)).
 *  - Calls that take a stream are asynchronous on it; a NULL stream is the
 *    legacy default stream.  One workspace serves one forward in flight.
 *  - Argument errors are reported synchronously, before anything is
 *    launched.  Launch failures return MOEFFN_ERR_CUDA.  Data-dependent
 *    errors found on the device (an expert id outside [-1, E), a bounded
 *    wait that ran out) are recorded in the workspace's status word and read
 *    with moeffn_get_device_status.
 */
#ifndef MOEFFN_H
#define MOEFFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOEFFN_ABI_VERSION 1

#if defined(__GNUC__)
#define MOEFFN_API __attribute__((visibility("default")))
#else
#define MOEFFN_API
#endif

typedef enum moeffn_status {
    MOEFFN_OK = 0,
    MOEFFN_ERR_INVALID_ARG = 1,          /* bad shape, null pointer, bad enum */
    MOEFFN_ERR_UNSUPPORTED = 2,          /* not an sm_103 device, or an option not built */
    MOEFFN_ERR_WORKSPACE_TOO_SMALL = 3,  /* a caller buffer is smaller than required */
    MOEFFN_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed */
    MOEFFN_ERR_TIMEOUT = 5,              /* a bounded device wait ran out (device status) */
    MOEFFN_ERR_OUT_OF_BOUNDS = 6         /* bounds-checked builds only (MOEFFN_BOUNDS_CHECK): a
                                            device index outside its buffer was caught and the
                                            access skipped (device status) */
} moeffn_status;

/* A cudaStream_t / CUstream handle passed through untouched. */
typedef void* moeffn_stream;

/* Problem description.  Limits checked by every call that takes it:
 *   num_tokens T >= 0; hidden H and intermediate I multiples of 128 (the
 *   UE8M0 packing granularity, as the MegaMoE host checks require);
 *   1 <= num_experts E <= 1024; 1 <= topk k <= min(E, 32).
 * act_clamp: optional activation clamp of the L1 epilogue (MegaMoE notes,
 *   "Activation clamp"; the pages' default threshold is 10): for c > 0 the
 *   BF16 gate value is clamped to <= c and the up value to [-c, c] before
 *   SwiGLU.  <= 0 disables it (the configs); NaN -> MOEFFN_ERR_INVALID_ARG.
 * fast_math: 0 = expf and a correctly rounded quotient in SiLU (Markstein's
 *   division method, checked bit for bit against IEEE division on the GPU for
 *   every BF16 input); 1 = approximate exponential and reciprocal (__expf,
 *   __fdividef), the pages' fast-math switch.  Other values return
 *   MOEFFN_ERR_UNSUPPORTED.
 * tile_n: most token rows per grouped-GEMM tile, a multiple of 16 in
 *   [32, 224]; 0 = 32 when T*k/E <= 32, 144 when T*k/E <= 272, else 224.
 *   Each expert's rows are split into ceil(n_e/tile_n) equal tiles rounded
 *   up to 16 rows.  For tile_n in [48, 144], when T*k > tile_n*E (an
 *   expert is expected to have more than one tile), that count is rounded
 *   up to an even number and the grouped GEMM stages each weight tile once
 *   for two token tiles of its expert (moeffn_paired_tiles).
 * wait_timeout_us: limit of every bounded device wait in microseconds;
 *   0 = 2 000 000 (2 s).
 * debug_flags: 0 for normal use.  Test hooks:
 *   bit 0 (MOEFFN_DEBUG_STARVE_L1): the L1 GEMM's load warp skips its first
 *     load, so the MMA warp's bounded wait runs out and the forward reports
 *     MOEFFN_ERR_TIMEOUT through the device status instead of hanging;
 *   bit 1 (MOEFFN_DEBUG_DUMP_L1_ACC): the forward stops after the L1 GEMM
 *     and leaves its raw FP32 accumulators in the output-pool view as
 *     float [P_max][2I] (gate channels 0..I-1, then up channels); needs
 *     4*I <= H, else MOEFFN_ERR_UNSUPPORTED; y is not written;
 *   bit 2 (MOEFFN_DEBUG_SPLIT_LAYERS): the grouped GEMM runs as two
 *     launches, all L1 items and then all L2 items, instead of one launch
 *     in which each L2 item waits for its token tile's L1 items; the
 *     results are the same bit for bit (per-layer timing, tests).
 * Pointers: x and y 16-byte aligned; prepared and workspace 256-byte
 * aligned; other arrays aligned to their element size (INVALID_ARG). */
typedef struct moeffn_problem {
    int32_t num_tokens;
    int32_t hidden;
    int32_t intermediate;
    int32_t num_experts;
    int32_t topk;
    float act_clamp;
    int32_t fast_math;
    int32_t tile_n;
    int32_t wait_timeout_us;
    int32_t debug_flags;
} moeffn_problem;

#define MOEFFN_DEBUG_STARVE_L1 1
#define MOEFFN_DEBUG_DUMP_L1_ACC 2
#define MOEFFN_DEBUG_SPLIT_LAYERS 4

/* Views into a workspace after moeffn_forward (for inspection and tests).
 * P_max = align(T*min(k,E) + E*127, 128) pool rows; P = offsets[E] <= P_max
 * rows are in use; NT_max = ceil(T*k/tile_n) + E token tiles (+ 2E instead
 * of + E when tiles are paired).  The n-th tile
 * of expert e has index tiles[e] + n and covers pool rows offsets[e] +
 * n*tile_rows[e] onwards.  Pool scale factors are stored per token tile and
 * per 128-wide K block as 256 uint32 words: word 128*h + 4*l + c holds the
 * packed scales of tile row 128*h + 32*c + l. */
typedef enum moeffn_view {
    MOEFFN_VIEW_STATUS = 0,     /* uint32 [16]: [0] error bits, [1] detail */
    MOEFFN_VIEW_COUNTS = 1,     /* int32 [E]: rows routed to each expert */
    MOEFFN_VIEW_OFFSETS = 2,    /* int32 [E+1]: first pool row of each expert, 128-row padded */
    MOEFFN_VIEW_TILES = 3,      /* int32 [E+1]: first token tile of each expert */
    MOEFFN_VIEW_SLOTS = 4,      /* int32 [T*k]: pool row of (t, j), -1 for an empty entry */
    MOEFFN_VIEW_ROW2TK = 5,     /* int32 [P_max]: t*k+j of a pool row, -1 for padding */
    MOEFFN_VIEW_WPOOL = 6,      /* float [P_max]: top-k weight of a pool row */
    MOEFFN_VIEW_SLACK = 7,      /* int32 [P_max/128]: padding rows per 128-row block */
    MOEFFN_VIEW_XPOOL = 8,      /* uint8 E4M3 [P_max][H]: gathered tokens */
    MOEFFN_VIEW_XPOOL_SF = 9,   /* uint32 [NT_max][H/128][256]: their scales (tile layout) */
    MOEFFN_VIEW_HPOOL = 10,     /* uint8 E4M3 [P_max][I]: requantised L1 output */
    MOEFFN_VIEW_HPOOL_SF = 11,  /* uint32 [NT_max][I/128][256]: its scales (tile layout) */
    MOEFFN_VIEW_YPOOL = 12,     /* uint16 BF16 [P_max][H]: L2 output per pool row */
    MOEFFN_VIEW_TILE_ROWS = 13  /* int32 [E]: token rows per tile of each expert */
} moeffn_view;

/* Human-readable name of a status code (host only; never NULL). */
MOEFFN_API const char* moeffn_status_string(moeffn_status status);

/* MOEFFN_ABI_VERSION of the loaded library (host only). */
MOEFFN_API int32_t moeffn_abi_version(void);

/* Validate a problem description against the limits above (host only). */
MOEFFN_API moeffn_status moeffn_check_problem(const moeffn_problem* problem);

/* Token tile rows the forward will use for this problem (host only). */
MOEFFN_API moeffn_status moeffn_tile_n(const moeffn_problem* problem, int32_t* tile_n);

/* 1 when the forward splits every expert into an even number of token tiles
 * whose pairs share each weight stage of the grouped GEMM, else 0 (host
 * only; the rule is under tile_n above). */
MOEFFN_API moeffn_status moeffn_paired_tiles(const moeffn_problem* problem, int32_t* paired);

/* Bytes of device workspace moeffn_forward needs (host only).  It holds the
 * schedule tables, the expert-sorted L1/L2 pools and their scales, and the
 * L2 output pool; its contents need no initialisation. */
MOEFFN_API moeffn_status moeffn_workspace_bytes(const moeffn_problem* problem, size_t* bytes);

/* Bytes of device memory for the prepared weights (host only). */
MOEFFN_API moeffn_status moeffn_prepared_weight_bytes(const moeffn_problem* problem, size_t* bytes);

/* Re-lay the expert weights for the grouped GEMMs (MegaMoE blog 7.3 "L1
 * weight interleave" and the SymmBuffer page's "transform_weights_for_mega_moe"
 * section: gate/up interleave and scale transpose for tensor-memory copy).
 *   w1     uint8 E2M1 [E][2I][H/2]  rows gate/up interleaved by 8
 *                                   (gate 0..7, up 0..7, gate 8..15, ...)
 *   w1_sf  uint32 UE8M0 [E][2I][H/128]
 *   w2     uint8 E2M1 [E][H][I/2]
 *   w2_sf  uint32 UE8M0 [E][H][I/128]
 *   prepared       device buffer of moeffn_prepared_weight_bytes bytes,
 *                  written by this call; opaque layout; must stay allocated
 *                  and unmodified while forwards use it.
 * Errors: null pointer -> INVALID_ARG; prepared_bytes too small ->
 * WORKSPACE_TOO_SMALL; not sm_103 -> UNSUPPORTED. */
MOEFFN_API moeffn_status moeffn_prepare_weights(const moeffn_problem* problem,
                                     const uint8_t* w1, const uint32_t* w1_sf,
                                     const uint8_t* w2, const uint32_t* w2_sf,
                                     void* prepared, size_t prepared_bytes,
                                     moeffn_stream stream);

/* Top-k routing (MegaMoE notes "Problem background": the router picks the
 * top-k experts of each token; the configs define it as softmax over the
 * router logits, top-k, weights renormalised over the selected experts).
 *   logits      float [T][E]; -inf allowed; a NaN logit ranks below every
 *               number (the pages leave NaN undefined; this is the reading
 *               the oracle follows too), so every id is valid and distinct
 *   topk_idx    int64 [T][k] out: experts by descending logit, ties to the
 *               lower expert index
 *   topk_w      float [T][k] out: exp(l_j - l_1) / sum_selected exp(l - l_1)
 * Errors: E > 1024, k > min(E, 32), null pointers -> INVALID_ARG. */
MOEFFN_API moeffn_status moeffn_route_topk(const float* logits, int32_t num_tokens, int32_t num_experts,
                                int32_t topk, int64_t* topk_idx, float* topk_w,
                                moeffn_stream stream);

/* The fused expert forward (MegaMoE notes "Execution overview", steps 2-9,
 * with the NVLink pull/push replaced by a local gather/scatter):
 *   x          uint8 E4M3 [T][H]
 *   x_sf       uint32 UE8M0 [T][H/128]
 *   topk_idx   int64 [T][k]; -1 marks an empty entry (skipped); other values
 *              outside [0, E) set a device error and are treated as -1
 *   topk_w     float [T][k]; applied in the L1 epilogue (h = silu(g) * u * w)
 *   prepared   output of moeffn_prepare_weights for this problem
 *   workspace  device buffer of moeffn_workspace_bytes bytes
 *   y          uint16 BF16 [T][H] out: sum over valid j of the BF16 L2 rows,
 *              accumulated in FP32 in j order, rounded to BF16 (RNE)
 * Errors: see the conventions above; workspace_bytes too small ->
 * WORKSPACE_TOO_SMALL.  T = 0 launches nothing.
 * Kernels: schedule tables, gather, ONE persistent grouped-GEMM launch (the
 * L1 items, then the L2 items, each L2 item waiting for the L1 items of its
 * token tile through GPU-scope counters: MegaMoE notes, "L1 -> L2
 * dependencies"), combine.  The GEMM launch sizes its grid to the CTA pairs
 * that can be resident at once and needs all of them resident together:
 * run the forward with the GPU to itself (another kernel holding SMs for
 * seconds would make the L2 items' bounded waits report a timeout).
 * On `stream` the call only launches kernels (the host checks arguments and
 * encodes tensor maps), so moeffn_route_topk and moeffn_forward can be
 * captured in a CUDA graph; a replay recomputes from what the buffers hold
 * then (tests/test_gpu_graph.py). */
MOEFFN_API moeffn_status moeffn_forward(const moeffn_problem* problem,
                             const uint8_t* x, const uint32_t* x_sf,
                             const int64_t* topk_idx, const float* topk_w,
                             const void* prepared, void* workspace, size_t workspace_bytes,
                             uint16_t* y, moeffn_stream stream);

/* moeffn_forward, additionally recording five caller-created CUDA events
 * (cudaEvent_t handles, same device) on `stream` at the stage boundaries:
 *   stage_events[0] before the schedule tables, [1] after the gather,
 *   [2] after the L1 GEMM, [3] after the L2 GEMM, [4] after the combine.
 *   The two layers run in one launch unless MOEFFN_DEBUG_SPLIT_LAYERS is
 *   set, so [2] and [3] are then recorded at the same point (after both).
 * Lets a caller time each stage with cudaEventElapsedTime.  A NULL array
 * or handle -> INVALID_ARG; otherwise errors as moeffn_forward. */
MOEFFN_API moeffn_status moeffn_forward_profiled(const moeffn_problem* problem,
                                                 const uint8_t* x, const uint32_t* x_sf,
                                                 const int64_t* topk_idx, const float* topk_w,
                                                 const void* prepared, void* workspace,
                                                 size_t workspace_bytes, uint16_t* y,
                                                 moeffn_stream stream, void* const* stage_events);

/* Device pointer and byte size of one view of a workspace (host only; no
 * GPU access).  Unknown view -> INVALID_ARG. */
MOEFFN_API moeffn_status moeffn_query(const moeffn_problem* problem, void* workspace, int32_t view,
                           void** dev_ptr, size_t* bytes);

/* Synchronise `stream`, then read the workspace status word written by the
 * last forward on it.  Returns MOEFFN_OK, MOEFFN_ERR_INVALID_ARG (an expert
 * id outside [-1, E) was seen) or MOEFFN_ERR_TIMEOUT (a bounded wait ran
 * out); *detail (optional) receives the raw status words [0] and [1].
 * Word [1] names the first wait that ran out: 1 a TMA producer (stage free),
 * 2 an MMA warp (accumulator drained), 3 an MMA warp (stage loaded),
 * 4 the epilogue (accumulator ready), 5 and 6 the end-of-kernel drains of
 * copies and MMAs, 7 a TMA producer waiting for the L1 rows of an L2 item's
 * token tile.  With a whole grid waiting on one failure, which of them
 * expires first is a race. */
MOEFFN_API moeffn_status moeffn_get_device_status(const moeffn_problem* problem, void* workspace,
                                       moeffn_stream stream, uint32_t* detail);

/* Allocation-free schedule tables.  The pages have no counterpart to this
 * call; it serves callers that cannot allocate device memory at the moment
 * they need the routing tables: servers that reserve their whole memory
 * budget at start-up and forbid later allocations, and latency-critical
 * loops that must not call cudaMalloc/cudaFree because those can
 * synchronise the device.  It computes the same counts, 128-row padded
 * offsets and (token, k) -> slot table as moeffn_forward (views COUNTS,
 * OFFSETS, SLOTS) with no workspace: its scratch is one static device array
 * of MOEFFN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library keeps until the process exits.
 *   topk_idx  int64 [T][k]; -1 = empty; other ids outside [0, E) are
 *             treated as empty (slot -1)
 *   counts    int32 [E] out;  offsets int32 [E+1] out;  slots int32 [T*k] out
 * Needs 64 + 4*T*k + 4*ceil(T*k/1024)*E bytes of the static scratch; larger
 * problems return MOEFFN_ERR_WORKSPACE_TOO_SMALL before anything runs.
 * Limits on T, E, k as moeffn_route_topk.  Allocates nothing and frees
 * nothing once the library is loaded on the device: with lazy module
 * loading (the CUDA default) the first call on a device loads the
 * library's device code, which reserves the array and may synchronise, so
 * make one call on each device at start-up, before any stream capture.
 * Every call looks up the array's device address with the calling thread's
 * current device.  All calls share the array and it keeps the last call's
 * contents: calls that overlap on the GPU race and give wrong tables. */
#define MOEFFN_NOALLOC_SCRATCH_BYTES (4u << 20)
MOEFFN_API moeffn_status moeffn_schedule_tables_noalloc(const int64_t* topk_idx, int32_t num_tokens,
                                                        int32_t num_experts, int32_t topk,
                                                        int32_t* counts, int32_t* offsets,
                                                        int32_t* slots, moeffn_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* MOEFFN_H */
