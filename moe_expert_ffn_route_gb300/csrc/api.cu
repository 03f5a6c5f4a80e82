// C ABI of the fused MoE expert forward: argument checks, buffer layouts,
// tensor-map encoding and the launch sequence on one stream.
//
// Host checks follow the MegaMoE host wrapper as the code-reading notes
// describe it ("Host wrapper: strict shape checks": recipe (1, 1, 32),
// SwiGLU only, W1 [E, 2I, H], W2 [E, H, I], H and I aligned to the scale
// packing, one architecture only).  Pool capacity follows the MegaMoE
// "pool capacity" formula with one rank and 128-row blocks:
// P_max = align(T*min(k,E) + E*(128-1), 128).
#include "moeffn.h"
#include "common.cuh"
#include "kernels.h"

#include <cudaTypedefs.h>
#include <string.h>

using namespace moeffn;

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct WsLayout {
    size_t status, counts, offsets, tiles, tile_rows, tile_rec, l1_done, slots, rank, hist, row2tk, wpool, slack;
    size_t xpool, xpool_sf, hpool, hpool_sf, ypool, total;
    int64_t P_max, NT_max, nchunks;
};

struct PrepLayout {
    size_t w1p, w1p_sf, w2p, w2p_sf, total;
};

moeffn_status check_problem(const moeffn_problem* p) {
    if (!p) return MOEFFN_ERR_INVALID_ARG;
    if (p->num_tokens < 0 || p->hidden <= 0 || p->intermediate <= 0) return MOEFFN_ERR_INVALID_ARG;
    if (p->hidden % 128 != 0 || p->intermediate % 128 != 0) return MOEFFN_ERR_INVALID_ARG;
    if (p->num_experts < 1 || p->num_experts > 1024) return MOEFFN_ERR_INVALID_ARG;
    if (p->topk < 1 || p->topk > p->num_experts || p->topk > 32) return MOEFFN_ERR_INVALID_ARG;
    if (p->tile_n != 0 && (p->tile_n % kTileQuantum != 0 || p->tile_n < 32 || p->tile_n > kMaxTileN))
        return MOEFFN_ERR_INVALID_ARG;
    if (p->wait_timeout_us < 0) return MOEFFN_ERR_INVALID_ARG;
    if (p->debug_flags & ~(MOEFFN_DEBUG_STARVE_L1 | MOEFFN_DEBUG_DUMP_L1_ACC | MOEFFN_DEBUG_SPLIT_LAYERS))
        return MOEFFN_ERR_INVALID_ARG;
    if ((p->debug_flags & MOEFFN_DEBUG_DUMP_L1_ACC) && 4 * p->intermediate > p->hidden)
        return MOEFFN_ERR_UNSUPPORTED;
    if (!(p->act_clamp <= 0.f || p->act_clamp > 0.f)) return MOEFFN_ERR_INVALID_ARG;   // NaN
    if (p->fast_math != 0 && p->fast_math != 1) return MOEFFN_ERR_UNSUPPORTED;
    // sizes used in 32-bit index arithmetic on the device
    const int64_t N = static_cast<int64_t>(p->num_tokens) * p->topk;
    if (N > (int64_t(1) << 26)) return MOEFFN_ERR_INVALID_ARG;
    if (static_cast<int64_t>(p->num_experts) * 2 * p->intermediate > (int64_t(1) << 30) ||
        static_cast<int64_t>(p->num_experts) * p->hidden > (int64_t(1) << 30))
        return MOEFFN_ERR_INVALID_ARG;
    return MOEFFN_OK;
}

// Most token rows per GEMM tile.  Each expert's rows are split into
// ceil(n_e / tile_n) equal tiles rounded up to 16 rows.  By default: 32 when
// an expert expects at most 32 rows (decode-sized batches: narrow stages,
// more of them in flight), 144 up to 272 expected rows (most experts then
// split in two tiles of at most 144 rows, and three accumulators fit in
// tensor memory), else kMaxTileN (the widest MMAs, fewest tiles).
int choose_tile_n(const moeffn_problem& p) {
    if (p.tile_n) return p.tile_n;
    const double m = static_cast<double>(p.num_tokens) * p.topk / p.num_experts;
    return m <= 32.0 ? 32 : m <= 272.0 ? 144 : kMaxTileN;
}

// Pairs of token tiles per weight stage (tile bounds of 48 to 144 rows) when
// an expert is expected to have more than one tile, T*k > tile_n*E: then each
// weight stage feeds two tiles of its expert.  With fewer rows per expert
// most experts would get two half tiles sharing one weight stream, where one
// tile per stage keeps two weight streams per SM pair in flight.
bool choose_paired(const moeffn_problem& p) {
    const int tile_n = choose_tile_n(p);
    return pairable_tile_n(tile_n) &&
           static_cast<int64_t>(p.num_tokens) * p.topk > static_cast<int64_t>(tile_n) * p.num_experts;
}

WsLayout ws_layout(const moeffn_problem& p) {
    WsLayout L{};
    const int64_t T = p.num_tokens, H = p.hidden, I = p.intermediate, E = p.num_experts, k = p.topk;
    const int64_t N = T * k;
    const int64_t kmin = k < E ? k : E;
    L.P_max = static_cast<int64_t>(align_up(static_cast<size_t>(T * kmin + E * (kPoolBlock - 1)), kPoolBlock));
    const int64_t bn = choose_tile_n(p);
    // ceil(n_e / bn) tiles per expert, rounded up to even when paired: fewer
    // than n_e / bn + 1 (+ 2 when paired) per expert with rows
    L.NT_max = (N + bn - 1) / bn + (choose_paired(p) ? 2 * E : E);
    L.nchunks = (N + 1023) / 1024;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 1024);
        return at;
    };
    L.status = take(sizeof(DevStatus));
    L.counts = take(4 * E);
    L.offsets = take(4 * (E + 1));
    L.tiles = take(4 * (E + 1));
    L.tile_rows = take(4 * E);
    L.tile_rec = take(32 * L.NT_max);
    L.l1_done = take(4 * L.NT_max);
    L.slots = take(4 * N);
    L.rank = take(4 * N);
    L.hist = take(4 * L.nchunks * E);
    L.row2tk = take(4 * L.P_max);
    L.wpool = take(4 * L.P_max);
    L.slack = take(4 * (L.P_max / kPoolBlock));
    L.xpool = take(static_cast<size_t>(L.P_max) * H);
    L.xpool_sf = take(static_cast<size_t>(L.NT_max) * (H / 128) * 1024);
    L.hpool = take(static_cast<size_t>(L.P_max) * I);
    L.hpool_sf = take(static_cast<size_t>(L.NT_max) * (I / 128) * 1024);
    L.ypool = take(static_cast<size_t>(L.P_max) * H * 2);
    L.total = o;
    return L;
}

PrepLayout prep_layout(const moeffn_problem& p) {
    PrepLayout L{};
    const size_t H = p.hidden, I = p.intermediate, E = p.num_experts;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 1024);
        return at;
    };
    L.w1p = take(E * 2 * I * H / 2);
    L.w1p_sf = take(E * (2 * I / 128) * (H / 128) * 512);
    L.w2p = take(E * H * I / 2);
    L.w2p_sf = take(E * (H / 128) * (I / 128) * 512);
    L.total = o;
    return L;
}

// Current device must be an sm_103 part; also returns its SM count.
moeffn_status check_device(int* num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOEFFN_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOEFFN_ERR_CUDA;
    if (major != 10 || minor != 3) return MOEFFN_ERR_UNSUPPORTED;
    if (num_sms && cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MOEFFN_ERR_CUDA;
    return MOEFFN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2-D K-major tile map: inner dimension K elements, `rows` rows, box of
// 128 K elements x box_rows rows, 128-byte swizzle.  fp4 = packed E2M1
// expanded to 16-byte-aligned groups in shared memory.
bool make_map(CUtensorMap* m, const void* base, uint64_t k, uint64_t rows, uint32_t box_rows, bool fp4) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {k, rows};
    const cuuint64_t strides[1] = {fp4 ? k / 2 : k};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Scale array read as rows of `row_words` 32-bit words, one row per box.
bool make_sf_map(CUtensorMap* m, const void* base, uint64_t row_words, uint64_t rows, uint32_t box_words) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {row_words, rows};
    const cuuint64_t strides[1] = {row_words * 4};
    const cuuint32_t box[2] = {box_words, 1};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

const char* moeffn_status_string(moeffn_status s) {
    switch (s) {
        case MOEFFN_OK: return "ok";
        case MOEFFN_ERR_INVALID_ARG: return "invalid argument";
        case MOEFFN_ERR_UNSUPPORTED: return "unsupported";
        case MOEFFN_ERR_WORKSPACE_TOO_SMALL: return "buffer too small";
        case MOEFFN_ERR_CUDA: return "CUDA error";
        case MOEFFN_ERR_TIMEOUT: return "device wait timed out";
        case MOEFFN_ERR_OUT_OF_BOUNDS: return "device index out of bounds";
    }
    return "unknown status";
}

int32_t moeffn_abi_version(void) { return MOEFFN_ABI_VERSION; }

moeffn_status moeffn_check_problem(const moeffn_problem* p) { return check_problem(p); }

moeffn_status moeffn_tile_n(const moeffn_problem* p, int32_t* tile_n) {
    const moeffn_status s = check_problem(p);
    if (s != MOEFFN_OK) return s;
    if (!tile_n) return MOEFFN_ERR_INVALID_ARG;
    *tile_n = choose_tile_n(*p);
    return MOEFFN_OK;
}

moeffn_status moeffn_paired_tiles(const moeffn_problem* p, int32_t* paired) {
    const moeffn_status s = check_problem(p);
    if (s != MOEFFN_OK) return s;
    if (!paired) return MOEFFN_ERR_INVALID_ARG;
    *paired = choose_paired(*p) ? 1 : 0;
    return MOEFFN_OK;
}

moeffn_status moeffn_workspace_bytes(const moeffn_problem* p, size_t* bytes) {
    const moeffn_status s = check_problem(p);
    if (s != MOEFFN_OK) return s;
    if (!bytes) return MOEFFN_ERR_INVALID_ARG;
    *bytes = ws_layout(*p).total;
    return MOEFFN_OK;
}

moeffn_status moeffn_prepared_weight_bytes(const moeffn_problem* p, size_t* bytes) {
    const moeffn_status s = check_problem(p);
    if (s != MOEFFN_OK) return s;
    if (!bytes) return MOEFFN_ERR_INVALID_ARG;
    *bytes = prep_layout(*p).total;
    return MOEFFN_OK;
}

moeffn_status moeffn_prepare_weights(const moeffn_problem* p, const uint8_t* w1, const uint32_t* w1_sf,
                                     const uint8_t* w2, const uint32_t* w2_sf, void* prepared,
                                     size_t prepared_bytes, moeffn_stream stream) {
    moeffn_status s = check_problem(p);
    if (s != MOEFFN_OK) return s;
    if (!w1 || !w1_sf || !w2 || !w2_sf || !prepared) return MOEFFN_ERR_INVALID_ARG;
    if (!aligned(w1, 16) || !aligned(w2, 16) || !aligned(w1_sf, 4) || !aligned(w2_sf, 4) || !aligned(prepared, 256))
        return MOEFFN_ERR_INVALID_ARG;
    const PrepLayout L = prep_layout(*p);
    if (prepared_bytes < L.total) return MOEFFN_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_device(nullptr)) != MOEFFN_OK) return s;
    uint8_t* b = static_cast<uint8_t*>(prepared);
    PrepareArgs a{w1, w1_sf, w2, w2_sf,
                  b + L.w1p, reinterpret_cast<uint32_t*>(b + L.w1p_sf),
                  b + L.w2p, reinterpret_cast<uint32_t*>(b + L.w2p_sf),
                  p->hidden, p->intermediate, p->num_experts};
    return launch_prepare(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MOEFFN_OK : MOEFFN_ERR_CUDA;
}

moeffn_status moeffn_route_topk(const float* logits, int32_t T, int32_t E, int32_t k, int64_t* idx, float* w,
                                moeffn_stream stream) {
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 32) return MOEFFN_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !idx || !w)) return MOEFFN_ERR_INVALID_ARG;
    moeffn_status s = check_device(nullptr);
    if (s != MOEFFN_OK) return s;
    return launch_route_topk(logits, T, E, k, idx, w, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MOEFFN_OK
               : MOEFFN_ERR_CUDA;
}

}  // extern "C"

namespace {

// The forward; when `ev` is non-null, ev[0..4] are recorded on the stream
// before the schedule tables, after the gather, after L1, after L2 and
// after the combine.
moeffn_status forward_impl(const moeffn_problem* p, const uint8_t* x, const uint32_t* x_sf,
                           const int64_t* topk_idx, const float* topk_w, const void* prepared, void* workspace,
                           size_t workspace_bytes, uint16_t* y, moeffn_stream stream, cudaEvent_t const* ev) {
    moeffn_status s = check_problem(p);
    if (s != MOEFFN_OK) return s;
    if (!prepared || !workspace) return MOEFFN_ERR_INVALID_ARG;
    if (p->num_tokens > 0 && (!x || !x_sf || !topk_idx || !topk_w || !y)) return MOEFFN_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(x_sf, 4) || !aligned(topk_idx, 8) ||
        !aligned(topk_w, 4) || !aligned(prepared, 256) || !aligned(workspace, 256))
        return MOEFFN_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*p);
    if (workspace_bytes < L.total) return MOEFFN_ERR_WORKSPACE_TOO_SMALL;
    int num_sms = 0;
    if ((s = check_device(&num_sms)) != MOEFFN_OK) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    if (cudaMemsetAsync(w + L.status, 0, sizeof(DevStatus), st) != cudaSuccess) return MOEFFN_ERR_CUDA;
    auto mark = [&](int i) { return !ev || cudaEventRecord(ev[i], st) == cudaSuccess; };
    if (p->num_tokens == 0) {
        for (int i = 0; i < 5; ++i)
            if (!mark(i)) return MOEFFN_ERR_CUDA;
        return MOEFFN_OK;
    }
    if (!mark(0)) return MOEFFN_ERR_CUDA;

    const int T = p->num_tokens, H = p->hidden, I = p->intermediate, E = p->num_experts, k = p->topk;
    const int tile_n = choose_tile_n(*p);
    DevStatus* status = reinterpret_cast<DevStatus*>(w + L.status);
    int* counts = reinterpret_cast<int*>(w + L.counts);
    int* offsets = reinterpret_cast<int*>(w + L.offsets);
    int* tiles = reinterpret_cast<int*>(w + L.tiles);
    int* tile_rows = reinterpret_cast<int*>(w + L.tile_rows);
    int* tile_rec = reinterpret_cast<int*>(w + L.tile_rec);
    int* slots = reinterpret_cast<int*>(w + L.slots);

    int* l1_done = reinterpret_cast<int*>(w + L.l1_done);
    const int paired = choose_paired(*p) ? 1 : 0;
    LayoutArgs la{x, x_sf, topk_idx, topk_w, T, H, E, k, tile_n, paired,
                  reinterpret_cast<int*>(w + L.hist), reinterpret_cast<int*>(w + L.rank), counts, offsets,
                  tiles, tile_rows, tile_rec, l1_done, slots, reinterpret_cast<int*>(w + L.row2tk), reinterpret_cast<float*>(w + L.wpool),
                  reinterpret_cast<int*>(w + L.slack), w + L.xpool, reinterpret_cast<uint32_t*>(w + L.xpool_sf),
                  status, static_cast<int>(L.P_max), static_cast<int>(L.NT_max)};
    if (launch_layout(la, st) != cudaSuccess || !mark(1)) return MOEFFN_ERR_CUDA;

    const PrepLayout PL = prep_layout(*p);
    const uint8_t* pb = static_cast<const uint8_t*>(prepared);
    GemmMaps m1, m2;
    const uint64_t kb1 = H / 128, kb2 = I / 128;
    if (!make_map(&m1.a, pb + PL.w1p, H, static_cast<uint64_t>(E) * 2 * I, 128, true) ||
        !make_map(&m2.a, pb + PL.w2p, I, static_cast<uint64_t>(E) * H, 128, true) ||
        !make_sf_map(&m1.sfa, pb + PL.w1p_sf, 128, static_cast<uint64_t>(E) * (2 * I / 128) * kb1, 128) ||
        !make_sf_map(&m2.sfa, pb + PL.w2p_sf, 128, static_cast<uint64_t>(E) * (H / 128) * kb2, 128) ||
        !make_sf_map(&m1.sfb_512, w + L.xpool_sf, 256, static_cast<uint64_t>(L.NT_max) * kb1, 128) ||
        !make_sf_map(&m1.sfb_1k, w + L.xpool_sf, 256, static_cast<uint64_t>(L.NT_max) * kb1, 256) ||
        !make_sf_map(&m2.sfb_512, w + L.hpool_sf, 256, static_cast<uint64_t>(L.NT_max) * kb2, 128) ||
        !make_sf_map(&m2.sfb_1k, w + L.hpool_sf, 256, static_cast<uint64_t>(L.NT_max) * kb2, 256))
        return MOEFFN_ERR_CUDA;
    for (int i = 0; i < kNumTokenBoxes; ++i)
        if (!make_map(&m1.b[i], w + L.xpool, H, L.P_max, 8 * (i + 1), false) ||
            !make_map(&m2.b[i], w + L.hpool, I, L.P_max, 8 * (i + 1), false))
            return MOEFFN_ERR_CUDA;

    GemmArgs g{};
    g.tiles = tiles;
    g.tile_rec = tile_rec;
    g.E = E;
    g.H = H;
    g.I = I;
    g.wpool = reinterpret_cast<const float*>(w + L.wpool);
    g.hpool = w + L.hpool;
    g.hpool_sf = w + L.hpool_sf;
    g.ypool = reinterpret_cast<uint16_t*>(w + L.ypool);
    g.status = status;
    g.timeout_ns = static_cast<uint64_t>(p->wait_timeout_us ? p->wait_timeout_us : 2000000) * 1000ull;
    g.debug_flags = p->debug_flags;
    g.act_clamp = p->act_clamp > 0.f ? p->act_clamp : 0.f;
    g.fast_math = p->fast_math;
    g.num_sms = num_sms;
    g.tile_n = tile_n;
    g.paired = paired;

    g.l1_done = l1_done;
    if (p->debug_flags & MOEFFN_DEBUG_DUMP_L1_ACC) {
        // L1 only: the raw accumulators are left in the output pool
        g.run_l1 = 1;
        g.run_l2 = 0;
        return launch_gemm(m1, m2, g, st) == cudaSuccess && mark(2) ? MOEFFN_OK : MOEFFN_ERR_CUDA;
    }
    if (p->debug_flags & MOEFFN_DEBUG_SPLIT_LAYERS) {
        // the two layers as two launches of the same kernel (the stream orders them)
        g.run_l1 = 1;
        g.run_l2 = 0;
        if (launch_gemm(m1, m2, g, st) != cudaSuccess || !mark(2)) return MOEFFN_ERR_CUDA;
        g.run_l1 = 0;
        g.run_l2 = 1;
        if (launch_gemm(m1, m2, g, st) != cudaSuccess || !mark(3)) return MOEFFN_ERR_CUDA;
    } else {
        // one persistent launch: every L2 item waits for the L1 items of its token tile
        g.run_l1 = 1;
        g.run_l2 = 1;
        if (launch_gemm(m1, m2, g, st) != cudaSuccess || !mark(2) || !mark(3)) return MOEFFN_ERR_CUDA;
    }

    if (launch_combine(reinterpret_cast<const uint16_t*>(w + L.ypool), slots, T, H, k, y, static_cast<int>(L.P_max),
                       status, st) != cudaSuccess ||
        !mark(4))
        return MOEFFN_ERR_CUDA;
    return MOEFFN_OK;
}

}  // namespace

extern "C" {

moeffn_status moeffn_forward(const moeffn_problem* p, const uint8_t* x, const uint32_t* x_sf,
                             const int64_t* topk_idx, const float* topk_w, const void* prepared, void* workspace,
                             size_t workspace_bytes, uint16_t* y, moeffn_stream stream) {
    return forward_impl(p, x, x_sf, topk_idx, topk_w, prepared, workspace, workspace_bytes, y, stream, nullptr);
}

moeffn_status moeffn_forward_profiled(const moeffn_problem* p, const uint8_t* x, const uint32_t* x_sf,
                                      const int64_t* topk_idx, const float* topk_w, const void* prepared,
                                      void* workspace, size_t workspace_bytes, uint16_t* y, moeffn_stream stream,
                                      void* const* stage_events) {
    if (!stage_events) return MOEFFN_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i)
        if (!stage_events[i]) return MOEFFN_ERR_INVALID_ARG;
    return forward_impl(p, x, x_sf, topk_idx, topk_w, prepared, workspace, workspace_bytes, y, stream,
                        reinterpret_cast<cudaEvent_t const*>(stage_events));
}

moeffn_status moeffn_query(const moeffn_problem* p, void* workspace, int32_t view, void** dev_ptr, size_t* bytes) {
    const moeffn_status s = check_problem(p);
    if (s != MOEFFN_OK) return s;
    if (!workspace || !dev_ptr || !bytes) return MOEFFN_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*p);
    const size_t T = p->num_tokens, H = p->hidden, I = p->intermediate, E = p->num_experts, k = p->topk;
    size_t off = 0, n = 0;
    switch (view) {
        case MOEFFN_VIEW_STATUS: off = L.status; n = sizeof(DevStatus); break;
        case MOEFFN_VIEW_COUNTS: off = L.counts; n = 4 * E; break;
        case MOEFFN_VIEW_OFFSETS: off = L.offsets; n = 4 * (E + 1); break;
        case MOEFFN_VIEW_TILES: off = L.tiles; n = 4 * (E + 1); break;
        case MOEFFN_VIEW_SLOTS: off = L.slots; n = 4 * T * k; break;
        case MOEFFN_VIEW_ROW2TK: off = L.row2tk; n = 4 * L.P_max; break;
        case MOEFFN_VIEW_WPOOL: off = L.wpool; n = 4 * L.P_max; break;
        case MOEFFN_VIEW_SLACK: off = L.slack; n = 4 * (L.P_max / kPoolBlock); break;
        case MOEFFN_VIEW_XPOOL: off = L.xpool; n = static_cast<size_t>(L.P_max) * H; break;
        case MOEFFN_VIEW_XPOOL_SF: off = L.xpool_sf; n = static_cast<size_t>(L.NT_max) * (H / 128) * 1024; break;
        case MOEFFN_VIEW_HPOOL: off = L.hpool; n = static_cast<size_t>(L.P_max) * I; break;
        case MOEFFN_VIEW_HPOOL_SF: off = L.hpool_sf; n = static_cast<size_t>(L.NT_max) * (I / 128) * 1024; break;
        case MOEFFN_VIEW_TILE_ROWS: off = L.tile_rows; n = 4 * E; break;
        case MOEFFN_VIEW_YPOOL: off = L.ypool; n = static_cast<size_t>(L.P_max) * H * 2; break;
        default: return MOEFFN_ERR_INVALID_ARG;
    }
    *dev_ptr = static_cast<uint8_t*>(workspace) + off;
    *bytes = n;
    return MOEFFN_OK;
}

moeffn_status moeffn_get_device_status(const moeffn_problem* p, void* workspace, moeffn_stream stream,
                                       uint32_t* detail) {
    const moeffn_status s = check_problem(p);
    if (s != MOEFFN_OK) return s;
    if (!workspace) return MOEFFN_ERR_INVALID_ARG;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOEFFN_ERR_CUDA;
    uint32_t words[2] = {0, 0};
    if (cudaMemcpy(words, static_cast<uint8_t*>(workspace) + ws_layout(*p).status, sizeof(words),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOEFFN_ERR_CUDA;
    if (detail) {
        detail[0] = words[0];
        detail[1] = words[1];
    }
    if (words[0] & DEV_ERR_BOUNDS) return MOEFFN_ERR_OUT_OF_BOUNDS;
    if (words[0] & DEV_ERR_TIMEOUT) return MOEFFN_ERR_TIMEOUT;
    if (words[0] & DEV_ERR_BAD_EXPERT) return MOEFFN_ERR_INVALID_ARG;
    return MOEFFN_OK;
}

}  // extern "C"
