// mk_abi.cu -- host side of libmk.so: argument validation, workspace layout, TMA
// tensor-map encoding and the launches behind the extern "C" entry points of mk.h.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "mk.h"
#include "mk_internal.h"

namespace {

thread_local char g_last_error[512] = "";

mk_status fail(mk_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

mk_status fail_cuda(cudaError_t e, const char *what) {
    return fail(MK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr double kRasterL2Budget = 32e6;   // tile-major: bytes of A rows (all ranks) resident per band
constexpr double kBandL2Budget = 24e6;     // rank-major: bytes of one rank's A rows resident per band
constexpr int64_t kRankMajorMinRows = 1024;  // default compute order: rank-major from this M on
constexpr int64_t kChainedOneSmMaxRows = 256; // chained mode: one-SM tiles up to this M (unless tile owners)
#ifndef MK_CHAIN_OWNER_MAX_ROWS
#define MK_CHAIN_OWNER_MAX_ROWS 256
#endif
constexpr int64_t kChainedOwnerMaxRows = MK_CHAIN_OWNER_MAX_ROWS; // chained mode: tile owners up to this M
constexpr double kAccumulatorL2Budget = 36e6; // accumulate mode: bytes of one band's fp32 accumulators
constexpr double kOperandHintBytes = 64e6;     // A rows of a band beyond which operand loads take no L2 hints
constexpr int64_t kAgBandRows = 4;             // AllGather + GEMM: 256-row tile rows per rank-major band
// Pause between an epilogue's 32-column store chunks: an eighth of one unit's MMA time at about
// 0.33 us per 64-deep k-block, at most 1 us (4 chunks per warp then take at most half a unit).
int unit_pace_ns(int64_t K) {
    const double unit_ns = static_cast<double>((K + MK_BK - 1) / MK_BK) * 330.0;
    const double pace = unit_ns / 8.0;
    return static_cast<int>(pace > 1000.0 ? 1000.0 : pace);
}

// The unfused GEMM launch and the role split (static or adaptive) are always paced. Chained and
// accumulate modes, whose epilogues also load or reduce in L2 and hold up the next rank's fold,
// are paced only when units are long (K_r >= 2048): pacing them measured faster at K_r = 3584
// and slower at K_r = 1024.
int epilogue_pace_ns(const mk_opts &o, int64_t Kr) {
    if (o.flags & MK_FLAG_NO_EPILOGUE_PACING) return 0;
    const int64_t kb = (Kr + MK_BK - 1) / MK_BK;
    if ((o.split_mode == MK_SPLIT_CHAINED || o.split_mode == MK_SPLIT_ACCUMULATE) && kb < 32) return 0;
    return unit_pace_ns(Kr);
}

constexpr double kTailL2Bytes = 64e6;        // partial tiles that stay in L2 until the end of a call
constexpr double kTailL2Bandwidth = 12e12;   // bytes/s the grid streams from L2
constexpr double kHbmEfficiency = 0.8;       // streaming fraction of the nominal HBM bandwidth

// Nominal HBM bandwidth of the current device (bytes/s) from its memory clock and bus width,
// scaled to what a streaming kernel reaches; cached per process.
double device_hbm_bandwidth() {
    static double cached = 0.0;
    if (cached > 0.0) return cached;
    int dev = 0, khz = 0, bits = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&khz, cudaDevAttrMemoryClockRate, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&bits, cudaDevAttrGlobalMemoryBusWidth, dev) == cudaSuccess && khz > 0 && bits > 0)
        cached = 2.0 * khz * 1e3 * bits / 8.0 * kHbmEfficiency;
    else
        cached = 6.5e12;
    return cached;
}

// Rows of compute tiles per band: the A rows that are live while a band is computed (one rank's
// in rank-major order, all P ranks' in tile-major order) should fit in a slice of L2 so that each
// B column streamed past them is reused by the whole band.
int auto_raster_group(bool pair, int P, int64_t Kr, int64_t row_tiles, bool rank_major) {
    const double per_row = static_cast<double>(rank_major ? 1 : P) * (pair ? 2 * MK_BM : MK_BM) *
                           static_cast<double>(Kr) * 2.0;
    const double budget = rank_major ? kBandL2Budget : kRasterL2Budget;
    int64_t g = per_row > 0 ? static_cast<int64_t>(budget / per_row) : row_tiles;
    if (g > row_tiles) g = row_tiles;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}
constexpr int kCtrlPeriodNs = 1000;
constexpr int kTileMajorReducePairs = 8;   // adaptive split, tile-major order: reduce-role units at the start

// Column slices per output tile's reduction: by default the smallest power of two (at most 8)
// that gives every role unit a reduce item (each item restarts the staged pipeline, so finer
// slices only pay while some units would otherwise get none); never more slices than the staged
// reducer has chunks in a tile (CH = 8 KiB per rank for P <= 8, else 4 KiB).
int choose_reduce_split(int requested, int64_t items, int role_units, int bn, int P, int partial_esize) {
    const int nch = MK_BM * bn * partial_esize / (P <= 8 ? 8192 : 4096);
    int s = requested;
    if (s <= 0) {
        s = 1;
        while (s < 8 && items * s < role_units) s *= 2;
    }
    return s < nch ? s : nch;
}

int choose_bn(int64_t N) { return N > 128 ? 256 : 128; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Geometry;
void choose_band_slices(bool pair, int P, int64_t M, int64_t N, int64_t Kr, int64_t rows, const Geometry &g,
                        int32_t *band_rows, int32_t *band_cols);

struct Geometry {
    int bn;
    int64_t tiles_m, tiles_n, num_tiles, num_units, num_kb;
    int64_t pair_tiles_m, num_pair_tiles, num_pair_units;
    size_t flags_off, partials_off, total;
};

bool make_geometry(int P, int64_t M, int64_t N, int64_t Kr, Geometry *g, int bn = 0) {
    if (P < 1 || P > MK_MAX_P || M < 0 || N < 0 || Kr < 0) return false;
    g->bn = bn > 0 ? bn : choose_bn(N);
    g->tiles_m = (M + MK_BM - 1) / MK_BM;
    g->tiles_n = (N + g->bn - 1) / g->bn;
    g->num_tiles = g->tiles_m * g->tiles_n;
    g->num_units = g->num_tiles * P;
    g->num_kb = (Kr + MK_BK - 1) / MK_BK;
    g->pair_tiles_m = (g->tiles_m + 1) / 2;
    g->num_pair_tiles = g->pair_tiles_m * g->tiles_n;
    g->num_pair_units = g->num_pair_tiles * P;
    g->flags_off = MK_WS_HEADER_BYTES;
    g->partials_off = align_up(g->flags_off + static_cast<size_t>(g->num_units) * sizeof(uint32_t), MK_WS_ALIGN);
    g->total = g->partials_off + static_cast<size_t>(g->num_units) * MK_BM * g->bn * sizeof(float);
    return true;
}

// Chained and accumulate modes, rank-major: the running sums (or accumulators) of the tiles that a
// rank pass covers must stay in L2 until the next rank's pass, so a pass covers at most
// kAccumulatorL2Budget bytes of them: G tile rows x W tile columns.  Each pass of a rank reads that
// rank's A rows of the G rows and B columns of the W columns, so over the call B is read once per
// band of G rows and A once per slice of W columns: pick the (G, W) within the budget that moves
// the fewest operand bytes (W = the whole width is the plain banded order).  At P = 8, M = N = 8192,
// K_r = 3584: 8 pair rows x 17 tile columns per pass, 6 x 470 MB of operand reads instead of
// 9 x 470 MB with 4-row full-width bands; at M = 16384, K_r = 1024: 1.6 GB instead of 2.4 GB.
// (Chained units that cover all P ranks of a tile keep no running sums in L2; their tile order is
// set after this, see run_rowparallel.)
void choose_band_slices(bool pair, int P, int64_t M, int64_t N, int64_t Kr, int64_t rows, const Geometry &g,
                        int32_t *band_rows, int32_t *band_cols) {
    const double tile_bytes = static_cast<double>(pair ? 2 * MK_BM : MK_BM) * g.bn * 4.0;
    const double a_bytes = static_cast<double>(P) * M * Kr * 2.0, b_bytes = static_cast<double>(P) * Kr * N * 2.0;
    double best = -1.0;
    int64_t best_g = 1, best_w = g.tiles_n;
    for (int64_t G = 1; G <= rows; ++G) {
        int64_t W = static_cast<int64_t>(kAccumulatorL2Budget / (G * tile_bytes));
        if (W < 1) break;
        if (W > g.tiles_n) W = g.tiles_n;
        const double cost = static_cast<double>((rows + G - 1) / G) * b_bytes +
                            static_cast<double>((g.tiles_n + W - 1) / W) * a_bytes;
        if (best < 0.0 || cost < best) {
            best = cost;
            best_g = G;
            best_w = W;
        }
    }
    *band_rows = static_cast<int32_t>(best_g);
    *band_cols = best_w >= g.tiles_n ? 0 : static_cast<int32_t>(best_w);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// bf16 row-major matrix rows x cols, TMA box {box_cols (inner), box_rows}, 128-byte swizzle,
// out-of-bounds elements filled with zero.
mk_status encode_2d(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols, int box_cols, int box_rows) {
    auto enc = encoder();
    if (!enc) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return MK_OK;
}


mk_status check_opts(const mk_opts *o) {
    if (o->split_mode < MK_SPLIT_ADAPTIVE || o->split_mode > MK_SPLIT_CHAINED)
        return fail(MK_ERR_INVALID_ARG, "split_mode %d out of range", o->split_mode);
    if (o->split_mode == MK_SPLIT_STATIC && o->comm_sms < 1)
        return fail(MK_ERR_INVALID_ARG, "static split needs comm_sms >= 1");
    if (o->comm_sms < 0) return fail(MK_ERR_INVALID_ARG, "comm_sms < 0");
    if (o->num_ctas < 0) return fail(MK_ERR_INVALID_ARG, "num_ctas < 0");
    if (o->raster_group < 0) return fail(MK_ERR_INVALID_ARG, "raster_group < 0");
    if (o->reduce_split < 0 || o->reduce_split > 64)
        return fail(MK_ERR_INVALID_ARG, "reduce_split %d outside [0, 64]", o->reduce_split);
    if (o->chain_ranks < 0 || o->chain_ranks > MK_MAX_P)
        return fail(MK_ERR_INVALID_ARG, "chain_ranks %d outside [0, %d]", o->chain_ranks, MK_MAX_P);
    if (o->trace_bytes && !o->trace) return fail(MK_ERR_INVALID_ARG, "trace_bytes without trace buffer");
    if (o->trace && !aligned16(o->trace)) return fail(MK_ERR_ALIGNMENT, "trace buffer not 16-byte aligned");
    if ((o->flags & MK_FLAG_BF16_PARTIALS) &&
        (o->split_mode == MK_SPLIT_ACCUMULATE || o->split_mode == MK_SPLIT_CHAINED))
        return fail(MK_ERR_INVALID_ARG, "MK_FLAG_BF16_PARTIALS needs partial tiles (adaptive, static or unfused split)");
    return MK_OK;
}

// Shared front half of the two row-parallel ops.
mk_status run_rowparallel(int op, int P, int64_t M, int64_t N, int64_t Kr, const void *const *A,
                          const void *const *B, void *const *C, mk_dtype out_dtype, void *ws, size_t ws_bytes,
                          const mk_opts *opts_in, void *stream) {
    g_last_error[0] = '\0';
    if (P < 1 || P > MK_MAX_P) return fail(MK_ERR_INVALID_ARG, "P=%d outside [1, %d]", P, MK_MAX_P);
    if (M < 0 || N < 0 || Kr < 0) return fail(MK_ERR_INVALID_ARG, "negative dimension");
    if (out_dtype != MK_BF16 && out_dtype != MK_F32) return fail(MK_ERR_INVALID_ARG, "unknown out_dtype");
    if (!A || !B || !C || !ws) return fail(MK_ERR_INVALID_ARG, "null pointer array or workspace");
    mk_opts o;
    mk_opts_default(&o);
    if (opts_in) o = *opts_in;
    mk_status st = check_opts(&o);
    if (st != MK_OK) return st;
    if (N % 8 || Kr % 8) return fail(MK_ERR_UNSUPPORTED_SHAPE, "N=%lld and K_per_rank=%lld must be multiples of 8",
                                     (long long)N, (long long)Kr);
    if (M > INT32_MAX || N > INT32_MAX || Kr > INT32_MAX)
        return fail(MK_ERR_UNSUPPORTED_SHAPE, "dimension above 2^31-1");
    if (op == MK_IOP_RS && M % P) return fail(MK_ERR_UNSUPPORTED_SHAPE, "M=%lld not divisible by P=%d", (long long)M, P);
    Geometry g;
    make_geometry(P, M, N, Kr, &g);
    if (g.num_units > INT32_MAX) return fail(MK_ERR_UNSUPPORTED_SHAPE, "too many tiles");
    if (M == 0 || N == 0) return MK_OK;   // nothing to read or write
    for (int r = 0; r < P; ++r) {
        if (!C[r]) return fail(MK_ERR_INVALID_ARG, "C[%d] is null", r);
        if (!aligned16(C[r])) return fail(MK_ERR_ALIGNMENT, "C[%d] not 16-byte aligned", r);
        if (Kr > 0) {
            if (!A[r] || !B[r]) return fail(MK_ERR_INVALID_ARG, "A[%d] or B[%d] is null", r, r);
            if (!aligned16(A[r]) || !aligned16(B[r])) return fail(MK_ERR_ALIGNMENT, "A[%d]/B[%d] not 16-byte aligned", r, r);
        }
    }
    if (reinterpret_cast<uintptr_t>(ws) % MK_WS_ALIGN) return fail(MK_ERR_ALIGNMENT, "workspace not 256-byte aligned");
    if (ws_bytes < g.total)
        return fail(MK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes, g.total);

    // Chained mode on a short M.  With a single 256-row band (M <= 256) one SM pair owns each
    // 256 x 128 tile: it computes the tile's P ranks one after the other and its epilogue keeps
    // the running sum in TMEM (the same additions in the same order), so no fold waits on another
    // block.  Measured at P = 8, N = 8192, K_r = 1024, M = 256 (us per call): tile owners 56.4,
    // SM-pair units of all 8 / 4 / 2 ranks of a 256 x 256 tile 64.1 / 62.2 / 60.2 (32 tiles
    // leave most pairs idle), the one-rank chain on one-SM tiles 60.  From M = 512 on the SM-pair
    // units of all P ranks take over: 66.6 us at M = 512 against 85.3 for the one-SM chain and
    // 100 for tile owners.  A caller that fixes the tile kind or the unit order at M <= 256 gets
    // the one-rank chain on one-SM tiles; a withheld unit (fault injection) gives one-rank units
    // at any M.
    const bool chain_owner = o.split_mode == MK_SPLIT_CHAINED && M <= kChainedOwnerMaxRows && o.debug_skip_unit < 0 &&
                             (o.flags & (MK_FLAG_SINGLE_SM_TILES | MK_FLAG_RANK_MAJOR | MK_FLAG_TILE_MAJOR)) == 0;
    const bool chained_short = o.split_mode == MK_SPLIT_CHAINED && M <= kChainedOneSmMaxRows && !chain_owner;
    const bool pair = (o.flags & MK_FLAG_SINGLE_SM_TILES) == 0 && !chained_short;
    if (chain_owner) make_geometry(P, M, N, Kr, &g, 128);   // the workspace check above used the default tiles
    int resident = 0;
    cudaError_t e = mk_max_persistent_ctas(g.bn, pair, &resident);
    if (e != cudaSuccess) return fail_cuda(e, "occupancy query");
    const int S = o.num_ctas > 0 ? o.num_ctas : resident;
    if (S > resident)
        return fail(MK_ERR_NOT_RESIDENT, "persistent grid of %d blocks cannot be co-resident (%d fit)", S, resident);
    if (pair && (S & 1)) return fail(MK_ERR_INVALID_ARG, "num_ctas=%d must be even with SM-pair tiles", S);
    if (S < (pair ? 4 : 2)) return fail(MK_ERR_INVALID_ARG, "num_ctas=%d too small for two roles", S);
    if (o.split_mode == MK_SPLIT_STATIC && o.comm_sms > S - (pair ? 2 : 1))
        return fail(MK_ERR_INVALID_ARG, "comm_sms=%d leaves no compute SMs in a grid of %d", o.comm_sms, S);
    // role units: blocks, or SM pairs (communication SMs are then counted in whole pairs)
    const int role_units = pair ? S / 2 : S;
    const int per_role = pair ? 2 : 1;

    MkParams p;
    memset(&p, 0, sizeof p);
    // B as given (K_r x N, 64-column boxes), or N x K_r with one box of this CTA's B rows per
    // K slice (all BN rows with one-SM tiles, BN/2 with SM pairs)
    p.b_nk = (o.flags & MK_FLAG_B_NK) ? 1 : 0;
    const int b_rows = pair ? g.bn / 2 : g.bn;
    for (int r = 0; r < P && Kr > 0; ++r) {
        st = encode_2d(&p.tmA[r], A[r], M, Kr, MK_BK, MK_BM);
        if (st != MK_OK) return st;
        st = p.b_nk ? encode_2d(&p.tmB[r], B[r], N, Kr, MK_BK, b_rows) : encode_2d(&p.tmB[r], B[r], Kr, N, 64, MK_BK);
        if (st != MK_OK) return st;
    }
    if (op == MK_IOP_RS) {
        for (int r = 0; r < P; ++r) p.out[r] = C[r];
        p.num_out = P;
    } else {
        int n = 0;
        for (int r = 0; r < P; ++r) {
            bool seen = false;
            for (int q = 0; q < n; ++q) seen = seen || (p.out[q] == C[r]);
            if (!seen) p.out[n++] = C[r];
        }
        p.num_out = n;
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    p.hdr = reinterpret_cast<MkWsHeader *>(wsb);
    p.flags = reinterpret_cast<uint32_t *>(wsb + g.flags_off);
    p.partials = reinterpret_cast<float *>(wsb + g.partials_off);
    p.trace = o.trace;
    p.trace_cap = static_cast<uint32_t>(o.trace_bytes / sizeof(mk_trace_record));
    p.skip_unit = o.debug_skip_unit;
    p.timeout_ns = o.wait_timeout_ns ? o.wait_timeout_ns : kDefaultTimeoutNs;
    p.P = P;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.Kr = static_cast<int32_t>(Kr);
    p.tiles_m = static_cast<int32_t>(g.tiles_m);
    p.tiles_n = static_cast<int32_t>(g.tiles_n);
    p.num_tiles = static_cast<int32_t>(g.num_tiles);
    p.num_units = static_cast<int32_t>(g.num_units);
    p.num_kb = static_cast<int32_t>(g.num_kb);
    p.pair_tiles_m = static_cast<int32_t>(g.pair_tiles_m);
    p.num_pair_tiles = static_cast<int32_t>(g.num_pair_tiles);
    p.num_pair_units = static_cast<int32_t>(g.num_pair_units);
    p.op = op;
    p.out_bf16 = out_dtype == MK_BF16;
    p.rows_per_shard = static_cast<int32_t>(M / P);
    {
        int nr = (o.comm_sms + per_role - 1) / per_role;
        if (nr > role_units - 1) nr = role_units - 1;
        p.static_nr = nr < 1 ? 1 : nr;
    }
    // Rank-major bands pay off once there are several bands; a short M has a single band, whose
    // tiles would all complete in the last 1/P of the GEMM, so it keeps the tile-major order.
    p.rank_major = (o.flags & MK_FLAG_TILE_MAJOR) ? 0 : (o.flags & MK_FLAG_RANK_MAJOR) ? 1 : (M >= kRankMajorMinRows);
    // Where the adaptive controller starts (the caller's count if given).  In rank-major order a
    // tile's ranks finish a band pass apart, so its partial tiles are read back from HBM whenever
    // it is reduced, and an SM that reduces during the GEMM only moves bytes the end of the call
    // would move at the same cost: the measured static sweeps are fastest with no reduce role,
    // so the controller starts there.  In tile-major order (short M) a tile's partials are
    // written back to back and reducing them while the GEMM runs hides a reduction that has too
    // few tiles to fill the grid at the end: the sweeps were fastest with 2 to 42 reduce SMs at
    // M = 256 and 512, so it starts with kTileMajorReducePairs.
    p.init_nr = o.comm_sms > 0 ? p.static_nr : p.rank_major ? 0 : (kTileMajorReducePairs < role_units - 1 ? kTileMajorReducePairs : role_units - 1);
    const int64_t order_rows = pair ? g.pair_tiles_m : g.tiles_m;
    p.raster_group = o.raster_group > 0 ? o.raster_group
                                        : auto_raster_group(pair, P, Kr, order_rows, p.rank_major != 0);
    if (o.split_mode == MK_SPLIT_ACCUMULATE || o.split_mode == MK_SPLIT_CHAINED) {
        // Accumulate and chained modes: rank-major bands sized so that the band's fp32
        // accumulator (running-sum) tiles stay in L2 while the P ranks add into them one after
        // the other (the tile-major order has the P ranks of a tile meet on the same lines at
        // the same time)
        p.rank_major = (o.flags & MK_FLAG_TILE_MAJOR) ? 0 : 1;
        if (o.raster_group <= 0) {
            const double row_bytes = static_cast<double>(pair ? 2 * MK_BM : MK_BM) * g.tiles_n * g.bn * 4.0;
            int64_t band = static_cast<int64_t>(kAccumulatorL2Budget / row_bytes);
            if (!p.rank_major) band = auto_raster_group(pair, P, Kr, order_rows, false);
            p.raster_group = static_cast<int32_t>(band < 1 ? 1 : band > order_rows ? order_rows : band);
        }
        // tile owners walk the tiles column by column, so that the owners of one column's tiles
        // read each B_r column block at about the same time
        if (chain_owner && o.raster_group <= 0) p.raster_group = static_cast<int32_t>(g.pair_tiles_m);
        if (p.rank_major && o.raster_group <= 0 && !chain_owner)
            choose_band_slices(pair, P, M, N, Kr, order_rows, g, &p.raster_group, &p.band_cols);
    }
    p.l2_hints = (o.flags & MK_FLAG_NO_L2_HINTS) ? 0 : 1;
    p.cooperative = (o.flags & MK_FLAG_NO_COOPERATIVE) ? 0 : 1;
    p.discard = (o.flags & MK_FLAG_KEEP_PARTIALS) ? 0 : 1;
    p.ctrl_period_ns = kCtrlPeriodNs;
    p.epi_pace_ns = epilogue_pace_ns(o, Kr);
    p.partial_bf16 = (o.flags & MK_FLAG_BF16_PARTIALS) ? 1 : 0;
    p.chain_owner = chain_owner ? 1 : 0;
    // Chained mode on SM pairs: consecutive ranks of a tile in one unit, computed back to back
    // into the two TMEM accumulators in turn, fold into the running sum there; it crosses L2
    // once per unit, and with all P ranks in one unit (the default) never.  Measured at P = 8
    // (ms per call, 2 / 4 / 8 ranks per unit): 16384 x 8192, K_r = 1024: 1.536 / 1.497 / 1.411;
    // 8192 x 8192, K_r = 1024: 0.791 / 0.766 / 0.752; 2048 x 4096, K_r = 512: 0.092 / 0.090 / 0.084;
    // 8192 x 8192, K_r = 3584: 2.241 / 2.218 / 2.231; 1024 x 8192, K_r = 1024: 0.120 / 0.124 / 0.122.
    // A withheld unit (the fault injection counts one-rank units) keeps one rank per unit.
    p.chain_ranks = (o.split_mode == MK_SPLIT_CHAINED && pair && !chain_owner && o.debug_skip_unit < 0)
                        ? (o.chain_ranks > 0 && o.chain_ranks < P ? o.chain_ranks : P)
                        : 1;
    if (p.chain_ranks > 1)
        p.num_pair_units = static_cast<int32_t>(g.num_pair_tiles * ((P + p.chain_ranks - 1) / p.chain_ranks));
    if (p.chain_ranks == P && P > 1 && p.rank_major && o.raster_group <= 0) {
        // Whole-tile units run every rank of a tile: the tiles in flight (one per SM pair) share
        // operands rank by rank, so they are kept to a block of about sqrt(pairs) tile rows by
        // pairs / rows columns.  Measured at P = 8, M = N = 8192, K_r = 3584: 8 x 10 runs 2.197 ms,
        // 9 x 9 2.207, 8 rows x 17 columns (the running-sum slices) 2.215.
        int32_t G = 1;
        while ((G + 1) * (G + 1) <= role_units) ++G;
        if (G > g.pair_tiles_m) G = static_cast<int32_t>(g.pair_tiles_m);
        const int64_t W = (role_units + G - 1) / G;
        p.raster_group = G;
        p.band_cols = W < g.tiles_n ? static_cast<int32_t>(W) : 0;
    }
    // Operand loads: A rows evict_last and B columns evict_first keep a band's A rows in L2 while
    // B streams past them.  A unit of several ranks reads the band's A rows of all its ranks;
    // where those exceed kOperandHintBytes they cannot stay in L2 until the band's next tiles, the
    // tiles in flight share B as much as A, and both are read with the normal policy.  Measured
    // with units of all 8 ranks (8-row bands): K_r = 3584, M = N = 8192 (117 MB of band A rows):
    // 3.98 against 5.1-5.3 GB of DRAM reads per call and 1.9 % faster (eight interleaved pairs
    // of runs); K_r = 1024, M = 4096 (34 MB): 0.41 against 0.50 GB and 0.7 % slower without hints.
    {
        const double band_a = static_cast<double>(p.raster_group) * (pair ? 2 * MK_BM : MK_BM) * Kr * 2.0 *
                               p.chain_ranks;
        p.op_hints = p.l2_hints && !(p.chain_ranks > 1 && band_a > kOperandHintBytes);
    }
    const int esize = p.partial_bf16 ? 2 : 4;
    p.red_split = choose_reduce_split(o.reduce_split, pair ? g.num_pair_tiles : g.num_tiles, role_units, g.bn, P,
                                      esize);
    // Where whole tiles give each role unit fewer than eight reduce items, half tiles spread the
    // end of the call's reduction more evenly: the role split measured 1.7, 1.5, 0.9 and 0.1 %
    // faster at M = 1024, 2048, 4096 and 8192 (P = 8, N = 8192, K_r = 1024; 1.7 to 13.5 whole
    // tiles per pair), and slower with quarter tiles or with half tiles at 27 tiles per pair.
    if (o.reduce_split <= 0 && p.red_split < 2 &&
        (pair ? g.num_pair_tiles : g.num_tiles) * p.red_split < 8 * static_cast<int64_t>(role_units))
        p.red_split = choose_reduce_split(2, pair ? g.num_pair_tiles : g.num_tiles, role_units, g.bn, P, esize);
    {
        // SM time of one reduce item when the whole grid reduces at the end of the call: the
        // item's partial bytes at the grid's share of memory bandwidth (L2 when every partial
        // tile of the call fits there, else HBM)
        const double item_bytes = static_cast<double>(MK_BM) * g.bn * esize * P / p.red_split;
        const double partials = static_cast<double>(g.num_tiles) * MK_BM * g.bn * esize * P;
        const double bw = partials <= kTailL2Bytes ? kTailL2Bandwidth : device_hbm_bandwidth();
        p.ctrl_tail_ns = static_cast<int32_t>(item_bytes * S / bw * 1e9);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (o.split_mode == MK_SPLIT_UNFUSED) {
        p.mode = MK_MODE_COMPUTE_ONLY;
        // The reduce kernel deals its items out statically: half tiles (two items per tile) ran
        // 0.6-1.4 % faster than whole tiles at P = 8, N = 8192, M = 4096 and 16384 (K_r = 1024)
        // and M = 8192 (K_r = 3584), where whole tiles already give every block 13 or more.
        p.red_split = choose_reduce_split(o.reduce_split, g.num_tiles, S, g.bn, P, esize);
        if (o.reduce_split <= 0 && p.red_split < 2)
            p.red_split = choose_reduce_split(2, g.num_tiles, S, g.bn, P, esize);
        e = mk_launch_persistent(p, g.bn, pair, S, s);
        if (e != cudaSuccess) return fail_cuda(e, "launch of the per-rank GEMM kernel");
        e = mk_launch_reduce(p, g.bn, S, s);
        if (e != cudaSuccess) return fail_cuda(e, "launch of the reduce kernel");
        return MK_OK;
    }
    if (o.split_mode == MK_SPLIT_ACCUMULATE || o.split_mode == MK_SPLIT_CHAINED) {
        p.mode = o.split_mode == MK_SPLIT_ACCUMULATE ? MK_MODE_ACCUMULATE : MK_MODE_CHAINED;
        e = mk_launch_persistent(p, g.bn, pair, S, s);
        return e == cudaSuccess ? MK_OK : fail_cuda(e, "launch of the accumulating GEMM kernel");
    }
    p.mode = o.split_mode == MK_SPLIT_STATIC ? MK_MODE_STATIC : MK_MODE_ADAPTIVE;
    e = mk_launch_persistent(p, g.bn, pair, S, s);
    if (e != cudaSuccess) return fail_cuda(e, "launch of the fused kernel");
    return MK_OK;
}

// AllGather + GEMM workspace: the header and one readiness flag per 128-row chunk of A (rounded
// up to whole 256-row pair tiles) and receiving rank.
size_t ag_workspace_bytes(const Geometry &g, int P) {
    return MK_WS_HEADER_BYTES + align_up(static_cast<size_t>(P) * 2 * g.pair_tiles_m * sizeof(uint32_t), MK_WS_ALIGN);
}

// First split of AllGather + GEMM (roles are fixed for the call): SMs for the copies in proportion
// to their share of the work, at per-SM rates measured on GB300 while the GEMM runs: about
// 30 GB/s of bulk copies (read once, written P times) against 11 TFLOP/s of bf16 MMA.  The copy
// rate is taken low on purpose: in rank-major order the first band's rows are all needed at
// once, so the copies should run well ahead of the compute.
int initial_copy_pairs(int role_units, int P, int64_t M, int64_t N, int64_t K) {
    const double copy = static_cast<double>(M) * K * 2.0 * (P + 1) / 30e9;
    const double gemm = static_cast<double>(P) * 2.0 * M * N * K / 11e12;
    int nr = static_cast<int>(role_units * copy / (copy + gemm) + 0.5);
    if (nr < 1) nr = 1;
    if (nr > role_units - 1) nr = role_units - 1;
    return nr;
}

mk_status run_allgather(int P, int64_t M, int64_t N, int64_t K, const void *const *A_shard, const void *const *B,
                        void *const *A_gathered, void *const *C, mk_dtype out_dtype, void *ws, size_t ws_bytes,
                        const mk_opts *opts_in, void *stream) {
    g_last_error[0] = '\0';
    if (P < 1 || P > MK_MAX_P) return fail(MK_ERR_INVALID_ARG, "P=%d outside [1, %d]", P, MK_MAX_P);
    if (M < 0 || N < 0 || K < 0) return fail(MK_ERR_INVALID_ARG, "negative dimension");
    if (out_dtype != MK_BF16 && out_dtype != MK_F32) return fail(MK_ERR_INVALID_ARG, "unknown out_dtype");
    if (!A_shard || !B || !C || !ws) return fail(MK_ERR_INVALID_ARG, "null pointer array or workspace");
    mk_opts o;
    mk_opts_default(&o);
    if (opts_in) o = *opts_in;
    mk_status st = check_opts(&o);
    if (st != MK_OK) return st;
    if (o.split_mode == MK_SPLIT_ACCUMULATE || o.split_mode == MK_SPLIT_CHAINED)
        return fail(MK_ERR_INVALID_ARG, "MK_SPLIT_ACCUMULATE and MK_SPLIT_CHAINED apply to GEMM + AllReduce and "
                    "GEMM + ReduceScatter");
    if (o.flags & MK_FLAG_BF16_PARTIALS)
        return fail(MK_ERR_INVALID_ARG, "MK_FLAG_BF16_PARTIALS applies to GEMM + AllReduce and GEMM + ReduceScatter");
    if (o.flags & MK_FLAG_B_NK)
        return fail(MK_ERR_INVALID_ARG, "MK_FLAG_B_NK applies to GEMM + AllReduce and GEMM + ReduceScatter");
    if (N % 8 || K % 8)
        return fail(MK_ERR_UNSUPPORTED_SHAPE, "N=%lld and K=%lld must be multiples of 8", (long long)N, (long long)K);
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return fail(MK_ERR_UNSUPPORTED_SHAPE, "dimension above 2^31-1");
    if (M % P) return fail(MK_ERR_UNSUPPORTED_SHAPE, "M=%lld not divisible by P=%d", (long long)M, P);
    int n_gather = 0;
    for (int r = 0; r < P && A_gathered; ++r) n_gather += A_gathered[r] != nullptr;
    if (n_gather != 0 && n_gather != P)
        return fail(MK_ERR_INVALID_ARG, "A_gathered must hold P buffers or none");
    const bool gather = n_gather == P;
    if (!gather && (M / P) % MK_BM)
        return fail(MK_ERR_UNSUPPORTED_SHAPE, "without gathered buffers each shard (M/P=%lld rows) must be a "
                    "multiple of %d rows", (long long)(M / P), MK_BM);
    Geometry g;
    make_geometry(P, M, N, K, &g);
    if (g.num_pair_units > INT32_MAX) return fail(MK_ERR_UNSUPPORTED_SHAPE, "too many tiles");
    if (M == 0 || N == 0) return MK_OK;
    for (int r = 0; r < P; ++r) {
        if (!C[r]) return fail(MK_ERR_INVALID_ARG, "C[%d] is null", r);
        if (!aligned16(C[r])) return fail(MK_ERR_ALIGNMENT, "C[%d] not 16-byte aligned", r);
        if (K > 0) {
            if (!A_shard[r] || !B[r]) return fail(MK_ERR_INVALID_ARG, "A_shard[%d] or B[%d] is null", r, r);
            if (!aligned16(A_shard[r]) || !aligned16(B[r]) || (gather && !aligned16(A_gathered[r])))
                return fail(MK_ERR_ALIGNMENT, "operand of rank %d not 16-byte aligned", r);
        }
    }
    if (reinterpret_cast<uintptr_t>(ws) % MK_WS_ALIGN) return fail(MK_ERR_ALIGNMENT, "workspace not 256-byte aligned");
    const size_t need = ag_workspace_bytes(g, P);
    if (ws_bytes < need) return fail(MK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes, need);

    int resident = 0;
    cudaError_t e = mk_max_persistent_ctas(g.bn, true, &resident);
    if (e != cudaSuccess) return fail_cuda(e, "occupancy query");
    const int S = o.num_ctas > 0 ? o.num_ctas : resident;
    if (S > resident)
        return fail(MK_ERR_NOT_RESIDENT, "persistent grid of %d blocks cannot be co-resident (%d fit)", S, resident);
    if (S & 1) return fail(MK_ERR_INVALID_ARG, "num_ctas=%d must be even with SM-pair tiles", S);
    if (S < 4) return fail(MK_ERR_INVALID_ARG, "num_ctas=%d too small for two roles", S);
    if (o.split_mode == MK_SPLIT_STATIC && o.comm_sms > S - 2)
        return fail(MK_ERR_INVALID_ARG, "comm_sms=%d leaves no compute SMs in a grid of %d", o.comm_sms, S);
    const int role_units = S / 2;

    MkParams p;
    memset(&p, 0, sizeof p);
    for (int r = 0; r < P && K > 0; ++r) {
        st = gather ? encode_2d(&p.tmA[r], A_gathered[r], M, K, MK_BK, MK_BM)
                    : encode_2d(&p.tmA[r], A_shard[r], M / P, K, MK_BK, MK_BM);
        if (st != MK_OK) return st;
        st = encode_2d(&p.tmB[r], B[r], K, N, 64, MK_BK);
        if (st != MK_OK) return st;
    }
    for (int r = 0; r < P; ++r) {
        p.out[r] = C[r];
        p.ag_src[r] = A_shard[r];
        p.ag_dst[r] = gather ? A_gathered[r] : nullptr;
    }
    p.num_out = P;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    p.hdr = reinterpret_cast<MkWsHeader *>(wsb);
    p.flags = reinterpret_cast<uint32_t *>(wsb + MK_WS_HEADER_BYTES);
    p.partials = nullptr;
    p.trace = o.trace;
    p.trace_cap = static_cast<uint32_t>(o.trace_bytes / sizeof(mk_trace_record));
    p.skip_unit = o.debug_skip_unit;
    p.timeout_ns = o.wait_timeout_ns ? o.wait_timeout_ns : kDefaultTimeoutNs;
    p.P = P;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.Kr = static_cast<int32_t>(K);
    p.tiles_m = static_cast<int32_t>(g.tiles_m);
    p.tiles_n = static_cast<int32_t>(g.tiles_n);
    p.num_tiles = static_cast<int32_t>(g.num_tiles);
    p.num_units = static_cast<int32_t>(g.num_units);
    p.num_kb = static_cast<int32_t>(g.num_kb);
    p.pair_tiles_m = static_cast<int32_t>(g.pair_tiles_m);
    p.num_pair_tiles = static_cast<int32_t>(g.num_pair_tiles);
    p.num_pair_units = static_cast<int32_t>(g.num_pair_units);
    p.op = MK_IOP_AG;
    p.out_bf16 = out_dtype == MK_BF16;
    p.rows_per_shard = static_cast<int32_t>(M / P);
    int nr = o.comm_sms > 0 ? (o.comm_sms + 1) / 2 : initial_copy_pairs(role_units, P, M, N, K);
    if (nr > role_units - 1) nr = role_units - 1;
    p.static_nr = p.init_nr = nr < 1 ? 1 : nr;
    // Rank-major bands by default, as for the row-parallel ops: each rank multiplies its own
    // gathered copy of A with its own B, and computing a band rank by rank streams each B once
    // per band instead of once per tile row (measured 12 % faster, fused and unfused alike).
    p.rank_major = (o.flags & MK_FLAG_TILE_MAJOR) ? 0 : 1;
    // each rank multiplies its own gathered copy of A (P copies live at once); without gathered
    // copies every rank reads the same shards
    if (o.raster_group > 0)
        p.raster_group = o.raster_group;
    else if (p.rank_major)
        p.raster_group = static_cast<int32_t>(g.pair_tiles_m < kAgBandRows ? (g.pair_tiles_m > 0 ? g.pair_tiles_m : 1)
                                                                            : kAgBandRows);
    else
        p.raster_group = auto_raster_group(true, gather ? P : 1, K, g.pair_tiles_m, false);
    p.discard = 0;
    p.ctrl_period_ns = kCtrlPeriodNs;
    // paced like the row-parallel role split (3.5 % faster fused at M = 8192, N = 3584, K = 4096)
    p.epi_pace_ns = (o.flags & MK_FLAG_NO_EPILOGUE_PACING) ? 0 : unit_pace_ns(K);
    p.ctrl_tail_ns = 0;   // unused: AllGather + GEMM fixes the roles for the call
    p.red_split = 1;
    p.l2_hints = (o.flags & MK_FLAG_NO_L2_HINTS) ? 0 : 1;
    p.op_hints = p.l2_hints;
    p.cooperative = (o.flags & MK_FLAG_NO_COOPERATIVE) ? 0 : 1;
    p.ag_gather = gather;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!gather) {
        p.mode = MK_MODE_COMPUTE_ONLY;   // nothing to move: the compute role reads the shards in place
        e = mk_launch_persistent(p, g.bn, true, S, s);
        return e == cudaSuccess ? MK_OK : fail_cuda(e, "launch of the GEMM kernel");
    }
    if (o.split_mode == MK_SPLIT_UNFUSED) {
        p.mode = MK_MODE_COMM_ONLY;      // baseline: gather every chunk, then one GEMM kernel
        e = mk_launch_persistent(p, g.bn, true, S, s);
        if (e != cudaSuccess) return fail_cuda(e, "launch of the gather kernel");
        p.mode = MK_MODE_COMPUTE_ONLY;
        p.ag_wait = 0;                   // stream order replaces the chunk flags
        e = mk_launch_persistent(p, g.bn, true, S, s);
        return e == cudaSuccess ? MK_OK : fail_cuda(e, "launch of the GEMM kernel");
    }
    // Roles stay fixed for the call (see the claim rules); adaptive mode uses the shape's split.
    p.mode = MK_MODE_STATIC;
    p.ag_wait = 1;
    e = mk_launch_persistent(p, g.bn, true, S, s);
    return e == cudaSuccess ? MK_OK : fail_cuda(e, "launch of the fused kernel");
}

// ------------------------------------------------------------------ Ring Attention
// bf16 3-D tensor {cols (inner), rows, planes}, row-major planes, box {64, box_rows, 1}, 128-byte
// swizzle; rows past the end of a plane read as zero.
mk_status encode_3d(CUtensorMap *map, const void *ptr, int64_t planes, int64_t rows, int64_t cols, int box_rows) {
    auto enc = encoder();
    if (!enc) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(planes)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, static_cast<cuuint64_t>(rows * cols) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (CUresult %d)", static_cast<int>(r));
    return MK_OK;
}

int64_t attn_kv_tiles(int64_t S) { return (S + 127) / 128; }

size_t attn_workspace_bytes(int P, int64_t H, int64_t S) {
    const int64_t nflags = static_cast<int64_t>(P) * (P - 1) * H * attn_kv_tiles(S);
    return MK_WS_HEADER_BYTES + align_up(static_cast<size_t>(nflags > 0 ? nflags : 1) * sizeof(uint32_t), MK_WS_ALIGN);
}

mk_status run_ring_attention(int P, int64_t H, int64_t S, int64_t d, const void *const *Q, const void *const *K,
                             const void *const *V, void *const *O, float *const *lse, void *const *kv_ring,
                             mk_dtype out_dtype, float scale, void *ws, size_t ws_bytes, const mk_opts *opts_in,
                             void *stream) {
    g_last_error[0] = '\0';
    if (P < 1 || P > MK_MAX_P) return fail(MK_ERR_INVALID_ARG, "P=%d outside [1, %d]", P, MK_MAX_P);
    if (H < 0 || S < 0 || d < 0) return fail(MK_ERR_INVALID_ARG, "negative dimension");
    if (out_dtype != MK_BF16 && out_dtype != MK_F32) return fail(MK_ERR_INVALID_ARG, "unknown out_dtype");
    if (!Q || !K || !V || !O || !ws) return fail(MK_ERR_INVALID_ARG, "null pointer array or workspace");
    if (!(scale >= 0.0f) || scale == INFINITY) return fail(MK_ERR_INVALID_ARG, "scale must be finite and >= 0");
    mk_opts o;
    mk_opts_default(&o);
    if (opts_in) o = *opts_in;
    mk_status st = check_opts(&o);
    if (st != MK_OK) return st;
    if (o.split_mode != MK_SPLIT_ADAPTIVE && o.split_mode != MK_SPLIT_STATIC && o.split_mode != MK_SPLIT_UNFUSED)
        return fail(MK_ERR_INVALID_ARG, "Ring Attention takes the adaptive, static or unfused split");
    if (o.flags & (MK_FLAG_BF16_PARTIALS | MK_FLAG_B_NK))
        return fail(MK_ERR_INVALID_ARG, "MK_FLAG_BF16_PARTIALS and MK_FLAG_B_NK apply to the GEMM operations");
    if (d != MK_ATTN_D) return fail(MK_ERR_UNSUPPORTED_SHAPE, "head dimension d=%lld (supported: %d)", (long long)d, MK_ATTN_D);
    if (H > INT32_MAX || S > INT32_MAX || H * S > INT32_MAX)
        return fail(MK_ERR_UNSUPPORTED_SHAPE, "H * S above 2^31-1");
    const int64_t nq = (S + 511) / 512;   // a query unit: 512 rows, four 128-row tiles over an SM pair
    if (H * P * nq > INT32_MAX || H * P * (P - 1) * attn_kv_tiles(S) > INT32_MAX)
        return fail(MK_ERR_UNSUPPORTED_SHAPE, "too many tiles");
    if (H == 0 || S == 0) return MK_OK;
    int n_lse = 0, n_ring = 0;
    for (int r = 0; r < P; ++r) {
        if (!Q[r] || !K[r] || !V[r] || !O[r]) return fail(MK_ERR_INVALID_ARG, "Q, K, V or O of rank %d is null", r);
        if (!aligned16(Q[r]) || !aligned16(K[r]) || !aligned16(V[r]) || !aligned16(O[r]))
            return fail(MK_ERR_ALIGNMENT, "Q, K, V or O of rank %d not 16-byte aligned", r);
        if (lse && lse[r]) {
            ++n_lse;
            if (reinterpret_cast<uintptr_t>(lse[r]) & 3u) return fail(MK_ERR_ALIGNMENT, "lse[%d] not 4-byte aligned", r);
        }
        if (kv_ring && kv_ring[r]) {
            ++n_ring;
            if (!aligned16(kv_ring[r])) return fail(MK_ERR_ALIGNMENT, "kv_ring[%d] not 16-byte aligned", r);
        }
    }
    if (n_lse != 0 && n_lse != P) return fail(MK_ERR_INVALID_ARG, "lse must hold P buffers or none");
    if (n_ring != 0 && n_ring != P) return fail(MK_ERR_INVALID_ARG, "kv_ring must hold P buffers or none");
    if (reinterpret_cast<uintptr_t>(ws) % MK_WS_ALIGN) return fail(MK_ERR_ALIGNMENT, "workspace not 256-byte aligned");
    const size_t need = attn_workspace_bytes(P, H, S);
    if (ws_bytes < need) return fail(MK_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes, need);
    const bool ring = n_ring == P && P > 1;

    int resident = 0;
    cudaError_t e = mk_attn_max_ctas(&resident);
    if (e != cudaSuccess) return fail_cuda(e, "occupancy query");
    if (resident < 2)
        return fail(MK_ERR_NOT_RESIDENT, "the attention kernel (%zu bytes of shared memory, %d threads) fits %d blocks "
                    "on this device", mk_attn_smem_bytes(), MK_ATTN_THREADS, resident);
    const int grid = o.num_ctas > 0 ? o.num_ctas : resident;
    if (grid > resident)
        return fail(MK_ERR_NOT_RESIDENT, "persistent grid of %d blocks cannot be co-resident (%d fit)", grid, resident);
    if (grid < 2 || (grid & 1)) return fail(MK_ERR_INVALID_ARG, "num_ctas=%d: the grid is SM pairs (even, >= 2)", grid);
    if (o.split_mode == MK_SPLIT_STATIC && o.comm_sms > grid - 2)
        return fail(MK_ERR_INVALID_ARG, "comm_sms=%d leaves no compute SMs in a grid of %d", o.comm_sms, grid);

    MkAttnParams p;
    memset(&p, 0, sizeof p);
    for (int r = 0; r < P; ++r) {
        if ((st = encode_3d(&p.tmQ[r], Q[r], H, S, d, 128)) != MK_OK) return st;
        if ((st = encode_3d(&p.tmK[r], K[r], H, S, d, 64)) != MK_OK) return st;
        if ((st = encode_3d(&p.tmV[r], V[r], H, S, d, 128)) != MK_OK) return st;
        if (ring) {
            const int64_t planes = static_cast<int64_t>(P - 1) * 2 * H;
            if ((st = encode_3d(&p.tmRK[r], kv_ring[r], planes, S, d, 64)) != MK_OK) return st;
            if ((st = encode_3d(&p.tmRV[r], kv_ring[r], planes, S, d, 128)) != MK_OK) return st;
        }
        p.k[r] = K[r];
        p.v[r] = V[r];
        p.ring[r] = ring ? kv_ring[r] : nullptr;
        p.out[r] = O[r];
        p.lse[r] = n_lse ? lse[r] : nullptr;
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    p.hdr = reinterpret_cast<MkWsHeader *>(wsb);
    p.flags = reinterpret_cast<uint32_t *>(wsb + MK_WS_HEADER_BYTES);
    p.timeout_ns = o.wait_timeout_ns ? o.wait_timeout_ns : kDefaultTimeoutNs;
    p.skip_copy = o.debug_skip_unit;
    const double sc = scale > 0.0f ? static_cast<double>(scale) : 1.0 / sqrt(static_cast<double>(d));
    p.scale_log2 = static_cast<float>(sc * 1.4426950408889634);
    p.P = P;
    p.H = static_cast<int32_t>(H);
    p.S = static_cast<int32_t>(S);
    p.nt = static_cast<int32_t>(attn_kv_tiles(S));
    p.nq = static_cast<int32_t>(nq);
    p.num_units = static_cast<int32_t>(H * P * nq);
    p.num_copies = ring ? static_cast<int32_t>(H * P * (P - 1) * attn_kv_tiles(S)) : 0;
    p.use_ring = ring ? 1 : 0;
    p.out_bf16 = out_dtype == MK_BF16;
    p.cooperative = (o.flags & MK_FLAG_NO_COOPERATIVE) ? 0 : 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!ring) {
        p.mode = MK_ATTN_COMPUTE_ONLY;
        e = mk_launch_attention(p, grid, s);
        return e == cudaSuccess ? MK_OK : fail_cuda(e, "launch of the attention kernel");
    }
    if (o.split_mode == MK_SPLIT_UNFUSED) {
        p.mode = MK_ATTN_COPY_ONLY;   // the KV forwarding of every step first, then the attention
        e = mk_launch_attention(p, grid, s);
        if (e != cudaSuccess) return fail_cuda(e, "launch of the KV forwarding kernel");
        p.mode = MK_ATTN_COMPUTE_ONLY;
        e = mk_launch_attention(p, grid, s);
        return e == cudaSuccess ? MK_OK : fail_cuda(e, "launch of the attention kernel");
    }
    p.mode = MK_ATTN_FUSED;
    // by default the compute blocks' own copy warps forward every tile; a static split adds
    // comm_sms whole communication blocks
    p.copy_ctas = o.split_mode == MK_SPLIT_STATIC ? (o.comm_sms + 1) / 2 * 2 : 0;   // whole SM pairs
    e = mk_launch_attention(p, grid, s);
    return e == cudaSuccess ? MK_OK : fail_cuda(e, "launch of the fused Ring Attention kernel");
}

}  // namespace

void mk_internal_set_error(const char *msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

size_t mk_internal_flags_bytes(int P, int64_t M, int64_t N, int64_t K_per_rank) {
    Geometry g;
    if (!make_geometry(P, M, N, K_per_rank, &g)) return 0;
    return g.partials_off - g.flags_off;
}

bool mk_internal_accumulator_region(int P, int64_t M, int64_t N, int64_t K_per_rank, size_t *offset, size_t *bytes) {
    Geometry g;
    if (!make_geometry(P, M, N, K_per_rank, &g)) return false;
    *offset = g.partials_off;
    *bytes = static_cast<size_t>(g.num_tiles) * MK_BM * g.bn * sizeof(float);
    return true;
}

extern "C" {

void mk_opts_default(mk_opts *o) {
    if (!o) return;
    memset(o, 0, sizeof *o);
    o->split_mode = MK_SPLIT_ADAPTIVE;
    o->comm_sms = 0;
    o->wait_timeout_ns = kDefaultTimeoutNs;
    o->trace = nullptr;
    o->trace_bytes = 0;
    o->num_ctas = 0;
    o->flags = 0;
    o->debug_skip_unit = -1;
    o->raster_group = 0;
    o->reduce_split = 0;
    o->chain_ranks = 0;
}

size_t mk_workspace_size(int op, int P, int64_t M, int64_t N, int64_t K_per_rank) {
    Geometry g;
    if (!make_geometry(P, M, N, K_per_rank, &g)) return 0;
    if (op == MK_OP_ALLREDUCE || op == MK_OP_REDUCESCATTER) return g.total;
    if (op == MK_OP_ALLGATHER_GEMM) return ag_workspace_bytes(g, P);
    return 0;
}

mk_status mk_gemm_allreduce(int P, int64_t M, int64_t N, int64_t K_per_rank, const void *const *A,
                            const void *const *B, void *const *C, mk_dtype out_dtype, void *ws, size_t ws_bytes,
                            const mk_opts *opts, void *cuda_stream) {
    return run_rowparallel(MK_IOP_AR, P, M, N, K_per_rank, A, B, C, out_dtype, ws, ws_bytes, opts, cuda_stream);
}

mk_status mk_gemm_reducescatter(int P, int64_t M, int64_t N, int64_t K_per_rank, const void *const *A,
                                const void *const *B, void *const *C_shard, mk_dtype out_dtype, void *ws,
                                size_t ws_bytes, const mk_opts *opts, void *cuda_stream) {
    return run_rowparallel(MK_IOP_RS, P, M, N, K_per_rank, A, B, C_shard, out_dtype, ws, ws_bytes, opts,
                           cuda_stream);
}

mk_status mk_allgather_gemm(int P, int64_t M, int64_t N, int64_t K, const void *const *A_shard,
                            const void *const *B, void *const *A_gathered, void *const *C, mk_dtype out_dtype,
                            void *ws, size_t ws_bytes, const mk_opts *opts, void *cuda_stream) {
    return run_allgather(P, M, N, K, A_shard, B, A_gathered, C, out_dtype, ws, ws_bytes, opts, cuda_stream);
}

size_t mk_ring_attention_workspace_size(int P, int64_t H, int64_t S, int64_t d) {
    if (P < 1 || P > MK_MAX_P || H < 0 || S < 0 || d < 0) return 0;
    return attn_workspace_bytes(P, H, S);
}

mk_status mk_ring_attention(int P, int64_t H, int64_t S, int64_t d, const void *const *Q, const void *const *K,
                            const void *const *V, void *const *O, float *const *lse, void *const *kv_ring,
                            mk_dtype out_dtype, float scale, void *ws, size_t ws_bytes, const mk_opts *opts,
                            void *cuda_stream) {
    return run_ring_attention(P, H, S, d, Q, K, V, O, lse, kv_ring, out_dtype, scale, ws, ws_bytes, opts, cuda_stream);
}

mk_status mk_status_check(void *ws, void *cuda_stream) {
    g_last_error[0] = '\0';
    if (!ws) return fail(MK_ERR_INVALID_ARG, "null workspace");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    MkWsHeader h;
    e = cudaMemcpy(&h, ws, 64, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e, "reading the workspace status");
    if (h.status == MK_OK) return MK_OK;
    const uint32_t zero = 0;
    e = cudaMemcpy(ws, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e, "clearing the workspace status");
    return fail(static_cast<mk_status>(h.status), "device reported %s (wait site %u, index %u)",
                mk_status_string(static_cast<mk_status>(h.status)), h.err_site, h.err_index);
}

const char *mk_status_string(mk_status s) {
    switch (s) {
        case MK_OK: return "ok";
        case MK_ERR_INVALID_ARG: return "invalid argument";
        case MK_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MK_ERR_ALIGNMENT: return "misaligned pointer";
        case MK_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MK_ERR_CUDA: return "CUDA error";
        case MK_ERR_TIMEOUT: return "device wait timed out";
        case MK_ERR_INTERNAL: return "internal error";
        case MK_ERR_NOT_RESIDENT: return "persistent grid not co-resident";
    }
    return "unknown status";
}

const char *mk_last_error(void) { return g_last_error; }

}  // extern "C"
