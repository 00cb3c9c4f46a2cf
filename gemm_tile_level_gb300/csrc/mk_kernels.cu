// mk_kernels.cu -- the persistent, role-specialised GEMM + reduction kernels for sm_103a and
// the standalone reduction kernel of the unfused baseline.
//
// Method (mKernel: Fast Multi-GPU, Multi-Node Fused Kernels; abstract, Figure 2, Table 3):
// one persistent kernel whose thread blocks take a compute role or a communication role.
// Compute blocks write each finished output tile to GPU memory and set a readiness flag
// (Figure 2, step 1); communication blocks observe the flags and reduce the ranks' tiles
// (step 2; here the P ranks are P partitions of one GPU's HBM, so "communication" is the
// fixed-order reduction of the P partial tiles and the write of the result or its row
// shard).  An on-GPU controller reads progress counters and publishes the target number of
// communication blocks (Figure 2, dashed arrow; Figure 7).
//
// Two compute-tile shapes share everything but the MMA issue:
//   mk_pair_kernel<BN>  (default): a cluster of two CTAs on two SMs computes one 256 x BN tile
//       with tcgen05.mma.cta_group::2 (M=256); each CTA stages only its 128 rows of A and its
//       BN/2 columns of B, so a 7-stage TMA ring fits and L2->SM bytes per FLOP drop by a third.
//   mk_persistent_kernel<BN>: one CTA computes a 128 x BN tile with cta_group::1.
// Warp roles in a block (352 threads):
//   warp 0   : work scheduler (pair: the even CTA claims for both) and TMA producer
//   warp 1   : one thread issues tcgen05.mma into one of two TMEM accumulators (pair: even CTA)
//   warps 2-9: tcgen05.ld the accumulator, store the fp32 partial tile of rank r into rank r's
//              workspace partition with coalesced 512-byte warp stores, release flag[tile][r];
//              or, for a reduce item, acquire flag[tile][0..P-1], stream the P partials through
//              the idle TMA ring with bulk copies, sum them in rank order 0..P-1 and write C or
//              the shard
//   warp 10  : the split controller (block 0, adaptive mode)
//
// Two more ways to form the sum use the compute blocks alone (no reduce role):
//   chained    : the reduce role's additions in its order, so the same bits, made where the
//                partials are produced.  On SM pairs a compute unit covers chain_ranks
//                consecutive ranks of a tile (all P by default), computed back to back into the
//                two TMEM accumulators; the epilogue adds the sum so far into each new
//                accumulator in place and writes the output after rank P-1 (chain_span).  With
//                fewer ranks per unit, or one-SM tiles, the unit of (tile, r) acquires
//                flag[tile][r-1] and adds to the running sum stored in the workspace
//                (chain_partial).  On a short M one SM pair owns each 256 x 128 tile and keeps
//                the running sum in TMEM next to the accumulators (owner_tile);
//   accumulate : the epilogue adds its accumulator into one fp32 tile with L2 reductions, and
//                the last of the P contributions writes the output (no fixed order).
//
// Failure handling: every wait is bounded.  A wait for another block's progress (readiness
// flags, the work gate, the controller watchdog) gives up after timeout_ns and raises
// MK_ERR_TIMEOUT plus a grid-wide abort; then every block stops claiming work, skips pending
// reductions, and drains its queued compute items so that no TMA load or MMA is in flight at
// exit.  Waits inside one block's (or pair's) pipeline only give up after 4 x timeout_ns.
#include <atomic>

#include "mk_internal.h"
#include "mk_ptx.cuh"
#include "mk_device.cuh"
#include "mk.h"

namespace mk {

enum { ITEM_END = 0, ITEM_COMPUTE = 1, ITEM_REDUCE = 2 };

#define MK_REDUCE_RING_BYTES (192u * 1024u)   // staging ring of the standalone reduce kernel

constexpr int WQ = 4;          // depth of the per-block work queue
constexpr int ACC = 2;         // TMEM accumulators per block

// One-SM tiles: 128 x BN per CTA, A 16 KiB + B BN/64 boxes of 8 KiB per 64-deep K slice.
template <int BN>
struct Cfg1 {
    static constexpr int A_BYTES = MK_BM * MK_BK * 2;
    static constexpr int B_BOX_BYTES = 64 * MK_BK * 2;
    static constexpr int B_BOXES = BN / 64;
    static constexpr int STAGE_BYTES = A_BYTES + B_BOXES * B_BOX_BYTES;
    static constexpr int STAGES = (BN == 256) ? 4 : 6;
    static constexpr int TMEM_COLS = ACC * BN;
    static constexpr int TILE_FLOATS = MK_BM * BN;
    static constexpr uint32_t IDESC = idesc_bf16_f32(MK_BM, BN);
};

// SM-pair tiles: 256 x BN per cluster; per CTA A 16 KiB + its BN/2 columns of B.
template <int BN>
struct Cfg2 {
    static constexpr int A_BYTES = MK_BM * MK_BK * 2;
    static constexpr int B_BOX_BYTES = 64 * MK_BK * 2;
    static constexpr int B_BOXES = BN / 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BOXES * B_BOX_BYTES;
    static constexpr int STAGES = (BN == 256) ? 7 : 8;
    // all of TMEM: two accumulators, and with BN = 128 a third region for a tile owner's
    // running sum (chained mode on a short M)
    static constexpr int TMEM_COLS = 512;
    static_assert(ACC * BN <= 512 && (BN == 256 || (ACC + 1) * BN <= 512), "TMEM columns");
    static constexpr int TILE_FLOATS = MK_BM * BN;
    static constexpr uint32_t IDESC = idesc_bf16_f32(2 * MK_BM, BN);
};

template <int STAGES>
struct SmemCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[ACC];
    uint64_t tempty[ACC];
    uint64_t wfull[WQ];
    uint64_t wempty[WQ];
    uint64_t drain;
    uint64_t rfull[4];      // reduce / copy staging: one per chunk in flight
    int2 items[WQ];
    uint32_t tmem_base;
    uint32_t epoch;
    int abort;
    uint32_t peer_issued;   // pair kernel: number of K-slice loads the odd CTA's producer issued
    uint32_t issued;        // number of K-slice loads this CTA's producer issued
    uint32_t epi_done;      // work items the epilogue group has finished (read by the scheduler)
};

// Grouped raster over a tiles_m x tiles_n grid: groups of G rows walked column by column, so
// that concurrently computed tiles share A rows and B columns in L2.
__device__ __forceinline__ void raster(int t, int tiles_m, int tiles_n, int G, int &tm, int &tn) {
    const int per_group = G * tiles_n;
    const int g = t / per_group;
    const int first_m = g * G;
    const int gsize = min(G, tiles_m - first_m);
    const int local = t - g * per_group;
    tm = first_m + local % gsize;
    tn = local / gsize;
}

// Rank entries per tile in the unit order: P, or the P ranks taken chain_ranks at a time (chained
// mode on SM pairs computes several consecutive ranks of a tile in one unit, see chain_span).
__device__ __forceinline__ int rank_groups(const MkParams &p) {
    return p.chain_ranks > 1 ? (p.P + p.chain_ranks - 1) / p.chain_ranks : p.P;
}

// Compute unit u -> (tile t in raster order, rank r).  Tile-major order visits the P ranks of a
// tile back to back.  Rank-major order cuts the tile rows into bands of G rows (G = raster_group)
// and computes a band for rank 0, then the same band for rank 1, and so on: while one rank's band
// is computed, L2 holds that rank's A rows of the band and each B column is read once per band,
// instead of all P ranks' operands competing for L2 at once.  `rows` is tiles_m, or pair_tiles_m
// for SM-pair tiles.
__device__ __forceinline__ void unit_tile(const MkParams &p, int rows, int u, int &t, int &r) {
    const int P = rank_groups(p);
    if (!p.rank_major) {
        t = u / P;
        r = u - t * P;
        return;
    }
    const int per_band = p.raster_group * p.tiles_n;
    const int b = u / (per_band * P);
    const int rem = u - b * per_band * P;
    const int bt = min(p.raster_group, rows - b * p.raster_group) * p.tiles_n;   // tiles in band b
    r = rem / bt;
    t = b * per_band + (rem - r * bt);
}

// Compute unit u -> (tile row `row` of `rows`, tile column tn, rank entry r: the rank, or the
// rank group with p.chain_ranks > 1).  With p.band_cols > 0 (chained and accumulate modes,
// rank-major) each band of raster_group tile rows is further cut into slices of band_cols tile
// columns, and the P ranks are computed slice by slice: a slice's
// running sums stay in L2 through its P rank passes while B is read once per band and A once per
// slice, instead of B once per (shorter) band.  Tiles run column by column inside a slice.
// Otherwise the order of unit_tile and raster.
__device__ __forceinline__ void unit_coords(const MkParams &p, int rows, int u, int &row, int &tn, int &r) {
    if (p.band_cols <= 0 || !p.rank_major) {
        int t;
        unit_tile(p, rows, u, t, r);
        raster(t, rows, p.tiles_n, p.raster_group, row, tn);
        return;
    }
    const int G = p.raster_group, W = p.band_cols, P = rank_groups(p);
    const int per_band = P * G * p.tiles_n;
    const int b = u / per_band;
    const int rem = u - b * per_band;
    const int gsize = min(G, rows - b * G);
    const int per_slice = P * gsize * W;
    const int c = rem / per_slice;
    const int rem2 = rem - c * per_slice;
    const int wsize = min(W, p.tiles_n - c * W);
    r = rem2 / (gsize * wsize);
    const int l = rem2 - r * (gsize * wsize);
    row = b * G + l % gsize;
    tn = c * W + l / gsize;
}

// SM-pair compute unit u -> (pair tile row sm, tile column tn, ranks r0 .. r0 + nr - 1).
__device__ __forceinline__ void unit_span(const MkParams &p, int u, int &sm, int &tn, int &r0, int &nr) {
    int e;
    unit_coords(p, p.pair_tiles_m, u, sm, tn, e);
    if (p.chain_ranks > 1) {
        r0 = e * p.chain_ranks;
        nr = min(p.chain_ranks, p.P - r0);
    } else {
        r0 = e;
        nr = 1;
    }
}

// One past the largest compute unit index that tile t consumes (its rank P-1 unit).
__device__ __forceinline__ uint32_t tile_units_end(const MkParams &p, int rows, uint32_t t) {
    if (!p.rank_major) return (t + 1) * static_cast<uint32_t>(p.P);
    const uint32_t per_band = static_cast<uint32_t>(p.raster_group * p.tiles_n);
    const uint32_t b = t / per_band;
    const uint32_t local = t - b * per_band;
    const uint32_t bt = static_cast<uint32_t>(min(p.raster_group, rows - static_cast<int>(b) * p.raster_group) *
                                              p.tiles_n);
    return b * per_band * static_cast<uint32_t>(p.P) + static_cast<uint32_t>(p.P - 1) * bt + local + 1;
}

// ------------------------------------------------------------------ work claiming
// Role of a role unit (a block, or an SM pair) for its next claim: reduce if its index is
// >= R - target (the target is published by the controller or fixed by the caller); once the
// compute queue is empty every role unit reduces.  Role unit 0 always computes while compute
// work remains.
//
// Deadlock freedom: a reduction of item i is queued only after every compute unit it consumes
// has been claimed (by anyone).  Each block works through its queue in claim order, so a
// reduction waits only on units claimed before it, which in turn wait only on items claimed
// earlier still: the wait-for relation follows claim order and has no cycle.
//
// A reduce-role unit claims the next item only when the units finished so far come within P of
// the last unit it consumes, so reducers do not park on items far ahead of the compute front.
// Reduce items follow the order in which tiles complete: tile index order for either unit order.
//
// units_done counts `done_per_unit` increments per compute unit (1 for one-SM tiles, 2 for an
// SM pair whose two CTAs each count their half).
struct ClaimGeom {
    uint32_t num_units;   // compute units (tile, rank)
    uint32_t num_items;   // reduce items (tiles, or tile pairs, times split)
    uint32_t role_index;  // this role unit
    uint32_t role_units;  // role units in the grid
    uint32_t done_per_unit;
    uint32_t split;       // reduce items per tile (column slices of its reduction)
    int rows;             // tile rows of the unit order (tiles_m, or pair_tiles_m)
};

__device__ bool wait_claimed(const Ctx &c, uint32_t need) {
    uint64_t t0 = 0;
    for (uint32_t spin = 0; spin != 0xFFFFFFFFu; ++spin) {
        if (ld_relaxed_gpu(&c.hdr->compute_next) >= need) return true;
        if (global_abort(c)) return false;
        if (t0 == 0) t0 = globaltimer();
        else if (globaltimer() - t0 > c.timeout_ns) break;
        __nanosleep(100);
    }
    raise_error(c, MK_ERR_TIMEOUT, SITE_CLAIMED, need);
    return false;
}

// `target` is the published target_nr as the caller last read it (0 = unpublished): the producer
// loads it while it streams the current unit, so that a claim costs one atomic round trip.
__device__ int2 claim_work(const MkParams &p, const Ctx &c, const ClaimGeom &g, bool &exhausted, uint32_t target) {
    MkWsHeader *h = c.hdr;
    const uint32_t P = static_cast<uint32_t>(p.P);
    uint64_t gate_t0 = 0;
    uint32_t gate_seen = 0xFFFFFFFFu;
    for (uint32_t spin = 0; spin != 0xFFFFFFFFu; ++spin) {
        if (global_abort(c)) return make_int2(ITEM_END, 0);
        if (p.mode == MK_MODE_COMPUTE_ONLY || p.mode == MK_MODE_ACCUMULATE || p.mode == MK_MODE_CHAINED) {
            const uint32_t u = atomicAdd(&h->compute_next, 1u);
            if (u >= g.num_units) return make_int2(ITEM_END, 0);
            if (static_cast<int64_t>(u) == p.skip_unit) continue;
            return make_int2(ITEM_COMPUTE, static_cast<int>(u));
        }
        if (p.op == MK_IOP_AG) {
            // AllGather + GEMM, roles fixed for the call: communication units claim chunk copies
            // (which depend on nothing) and, once every copy is claimed, help compute; compute
            // units never claim copies.  A compute item then waits only on copies queued ahead of
            // every compute item of their block, so the wait-for relation has no cycle.
            if (p.mode == MK_MODE_COMM_ONLY || static_cast<int>(g.role_index) >= static_cast<int>(g.role_units) - p.static_nr) {
                const uint32_t i = atomicAdd(&h->reduce_next, 1u);
                if (i < g.num_items) return make_int2(ITEM_REDUCE, static_cast<int>(i));
                if (p.mode == MK_MODE_COMM_ONLY) return make_int2(ITEM_END, 0);
            }
            const uint32_t u = atomicAdd(&h->compute_next, 1u);
            if (u >= g.num_units) return make_int2(ITEM_END, 0);
            if (static_cast<int64_t>(u) == p.skip_unit) continue;
            return make_int2(ITEM_COMPUTE, static_cast<int>(u));
        }
        if (!exhausted) {
            int nr = p.static_nr;
            if (p.mode == MK_MODE_ADAPTIVE) nr = target ? static_cast<int>(target) - 1 : p.init_nr;   // target + 1
            if (static_cast<int>(g.role_index) < static_cast<int>(g.role_units) - nr) {
                const uint32_t u = atomicAdd(&h->compute_next, 1u);
                if (u < g.num_units) {
                    if (static_cast<int64_t>(u) == p.skip_unit) continue;
                    return make_int2(ITEM_COMPUTE, static_cast<int>(u));
                }
                exhausted = true;
            } else {
                const uint32_t next = ld_relaxed_gpu(&h->reduce_next);
                if (next >= g.num_items) return make_int2(ITEM_END, 0);
                const uint32_t done = ld_relaxed_gpu(&h->units_done);
                const uint32_t issued = ld_relaxed_gpu(&h->compute_next);
                const uint64_t slack = static_cast<uint64_t>(P) * g.done_per_unit;
                const uint64_t need = tile_units_end(p, g.rows, next / g.split);
                if (issued < g.num_units && need * g.done_per_unit > done + slack) {
                    // nothing ready yet: wait for compute progress (bounded), then re-read the role
                    if (done != gate_seen) {
                        gate_seen = done;
                        gate_t0 = globaltimer();
                    } else if (globaltimer() - gate_t0 > c.timeout_ns) {
                        raise_error(c, MK_ERR_TIMEOUT, SITE_GATE, next);
                        return make_int2(ITEM_END, 0);
                    }
                    __nanosleep(200);
                    continue;
                }
            }
        }
        const uint32_t i = atomicAdd(&h->reduce_next, 1u);
        if (i >= g.num_items) return make_int2(ITEM_END, 0);
        const uint64_t need64 = tile_units_end(p, g.rows, i / g.split);
        const uint32_t need = need64 < g.num_units ? static_cast<uint32_t>(need64) : g.num_units;
        if (!wait_claimed(c, need)) return make_int2(ITEM_END, 0);
        return make_int2(ITEM_REDUCE, static_cast<int>(i));
    }
    raise_error(c, MK_ERR_TIMEOUT, SITE_GATE, 0);
    return make_int2(ITEM_END, 0);
}

// A block that has just queued a compute unit claims the next one with one atomic before it loads
// the current unit, so that the atomic's round trip overlaps those loads instead of falling
// between the last load of one unit and the first load of the next (only STAGES k-slices are
// buffered ahead of the MMA).  The unit claimed ahead is always the block's next item, whatever
// role the controller publishes meanwhile, so the wait-for relation still follows claim order.
constexpr uint32_t NO_CLAIM = 0xFFFFFFFFu;

__device__ __forceinline__ bool claims_ahead(const MkParams &p) {
    return p.op != MK_IOP_AG && p.mode != MK_MODE_COMM_ONLY;
}

// The work item for unit `u`, claimed ahead (see claims_ahead).  Past the last unit, the role
// split goes on to reduce items; the other modes have nothing left.
__device__ int2 item_claimed_ahead(const MkParams &p, const Ctx &c, const ClaimGeom &g, uint32_t u, bool &exhausted,
                                   uint32_t target) {
    if (global_abort(c)) return make_int2(ITEM_END, 0);
    if (u >= g.num_units) {
        if (p.mode != MK_MODE_ADAPTIVE && p.mode != MK_MODE_STATIC) return make_int2(ITEM_END, 0);
        exhausted = true;
        return claim_work(p, c, g, exhausted, target);
    }
    if (static_cast<int64_t>(u) == p.skip_unit) return claim_work(p, c, g, exhausted, target);
    return make_int2(ITEM_COMPUTE, static_cast<int>(u));
}

// ------------------------------------------------------------------ reduction of one tile
__device__ __forceinline__ void store_out4(const MkParams &p, int grow, int gcol, float4 v) {
    if (p.op == MK_IOP_RS) {
        const int sh = grow / p.rows_per_shard;
        const int lr = grow - sh * p.rows_per_shard;
        const size_t idx = static_cast<size_t>(lr) * p.N + gcol;
        if (p.out_bf16)
            st_u2(static_cast<uint16_t *>(p.out[sh]) + idx, pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
        else
            st_f4(static_cast<float *>(p.out[sh]) + idx, v.x, v.y, v.z, v.w);
    } else {
        const size_t idx = static_cast<size_t>(grow) * p.N + gcol;
        for (int d = 0; d < p.num_out; ++d) {
            if (p.out_bf16)
                st_u2(static_cast<uint16_t *>(p.out[d]) + idx, pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
            else
                st_f4(static_cast<float *>(p.out[d]) + idx, v.x, v.y, v.z, v.w);
        }
    }
}

// Partial tile (rank r, tile (tm, tn)) lives at ((r * num_tiles) + tm * tiles_n + tn) tiles into
// the partial region.  Inside a tile the layout is 16-byte column groups, [group][128 rows]:
// four floats per group for fp32 partials, eight bf16 for bf16 partials (MK_FLAG_BF16_PARTIALS).
template <int BN>
__device__ __forceinline__ uint32_t partial_tile_bytes(const MkParams &p) {
    return MK_BM * BN * (p.partial_bf16 ? 2u : 4u);
}

template <int BN>
__device__ __forceinline__ char *partial_tile_at(const MkParams &p, int r, int lt) {
    return reinterpret_cast<char *>(p.partials) +
           (static_cast<size_t>(r) * p.num_tiles + lt) * partial_tile_bytes<BN>(p);
}

// fp32 tiles (chained running sums, accumulate mode, which never store bf16 partials)
template <int BN>
__device__ __forceinline__ float *partial_tile(const MkParams &p, int r, int lt) {
    return p.partials + (static_cast<size_t>(r) * p.num_tiles + lt) * (MK_BM * BN);
}

// Chunks [c0, c1) of a partial tile that reduce slice `sub` of `nsub` covers: whole chunks of the
// staged reduction (CH bytes per rank, see reduce_tile_staged).
template <int BN>
__device__ __forceinline__ void slice_chunks(const MkParams &p, int sub, int nsub, uint32_t &c0, uint32_t &c1,
                                             uint32_t &ch_bytes) {
    ch_bytes = p.P <= 8 ? 8192u : 4096u;
    const uint32_t nch = partial_tile_bytes<BN>(p) / ch_bytes;
    c0 = static_cast<uint32_t>(sub) * nch / static_cast<uint32_t>(nsub);
    c1 = static_cast<uint32_t>(sub + 1) * nch / static_cast<uint32_t>(nsub);
}

// Drop the consumed part (slice sub of nsub) of the partial tiles of tile lt from L2 without
// write-back (scratch data).
template <int BN>
__device__ __forceinline__ void discard_tile(const MkParams &p, int lt, int sub, int nsub, int tid, int nthreads) {
    uint32_t c0, c1, chb;
    slice_chunks<BN>(p, sub, nsub, c0, c1, chb);
    const int l0 = static_cast<int>(c0 * chb / 128), l1 = static_cast<int>(c1 * chb / 128);
    for (int r = 0; r < p.P; ++r) {
        const char *base = partial_tile_at<BN>(p, r, lt);
        for (int l = l0 + tid; l < l1; l += nthreads) discard_l2_line(base + static_cast<size_t>(l) * 128);
    }
}

// The first warp of the reduce group: lane r acquires flag[lt][r] == epoch, all P flags polled at
// once (one round trip per poll instead of P).  Every lane returns the same value: false if the
// grid is aborting or the limit ran out (which raises MK_ERR_TIMEOUT).
__device__ bool wait_tile_ready(const MkParams &p, const Ctx &c, int lt, uint32_t epoch, int lane) {
    const uint32_t *f = p.flags + static_cast<size_t>(lt) * p.P;
    bool seen = lane >= p.P;
    uint64_t t0 = 0;
    for (uint32_t polls = 0;; ++polls) {
        if (!seen) seen = ld_acquire_gpu(f + lane) == epoch;
        if (__all_sync(0xFFFFFFFFu, seen)) return true;
        int stop = 0;
        if (lane == 0) {
            if (*c.s_abort) {
                stop = 1;
            } else {
                if (t0 == 0) t0 = globaltimer();
                if ((polls & 15u) == 15u) {
                    if (global_abort(c)) {
                        stop = 1;
                    } else if (globaltimer() - t0 > c.timeout_ns || polls > (1u << 30)) {
                        raise_error(c, MK_ERR_TIMEOUT, SITE_FLAG, static_cast<uint32_t>(lt * p.P));
                        stop = 1;
                    }
                }
            }
        }
        if (__shfl_sync(0xFFFFFFFFu, stop, 0)) return false;
        __nanosleep(32);
    }
}

// Reduce-role staging through the block's TMA ring, which is idle while the block reduces (the
// producer reloads it only after the epilogue group has finished its last reduce item).
struct Staging {
    uint8_t *ring;          // 1024-byte aligned, ring_bytes long
    uint32_t ring_bytes;
    uint64_t *rfull;        // 3 mbarriers, one per chunk set in flight
    uint32_t seq;           // chunk sets consumed so far by this block (phase bookkeeping)
};

// Eight fp32 values (columns gcol..gcol+7 of row grow) of the result, AllReduce or shard.
__device__ __forceinline__ void store_out8(const MkParams &p, int grow, int gcol, float4 a, float4 b) {
    void *base;
    size_t idx;
    int nout = 1;
    if (p.op == MK_IOP_RS) {
        const int sh = grow / p.rows_per_shard;
        base = p.out[sh];
        idx = static_cast<size_t>(grow - sh * p.rows_per_shard) * p.N + gcol;
    } else {
        base = p.out[0];
        idx = static_cast<size_t>(grow) * p.N + gcol;
        nout = p.num_out;
    }
    for (int d = 0; d < nout; ++d) {
        void *o = d == 0 ? base : p.out[d];
        if (p.out_bf16) {
            st_u4(static_cast<uint16_t *>(o) + idx, pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                  pack_bf16x2(b.z, b.w));
        } else {
            st_f4(static_cast<float *>(o) + idx, a.x, a.y, a.z, a.w);
            st_f4(static_cast<float *>(o) + idx + 4, b.x, b.y, b.z, b.w);
        }
    }
}

// Eight packed bf16 (element 0 in the low half of word 0) to fp32, exactly.
__device__ __forceinline__ void widen_bf16x8(uint4 w, float4 &lo, float4 &hi) {
    lo = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                     __uint_as_float(w.y & 0xFFFF0000u));
    hi = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u), __uint_as_float(w.w << 16),
                     __uint_as_float(w.w & 0xFFFF0000u));
}

// Sum the P partial tiles of tile (tm, tn) in rank order r = 0..P-1, over column slice `sub` of
// `nsub` (a reduce item covers one slice, so that a few large tiles still spread over many SMs).
// The tiles are streamed in chunks of CH bytes per rank (chunk c = column groups
// [c*CH/2048, ...) x 128 rows) by bulk copies into the ring, up to three chunk sets (P x CH bytes
// each) in flight, so each SM keeps up to 192 KiB of loads outstanding without holding them in
// registers.  Thread etid owns row etid % 128 and two column groups (eight columns) of every
// 8 KiB chunk (one group of a 4 KiB chunk when P > 8), read conflict-free from shared memory.
template <int BN>
__device__ void reduce_tile_staged(const MkParams &p, const Ctx &c, int tm, int tn, int sub, int nsub, int etid,
                                   Staging &st) {
    const int lt = tm * p.tiles_n + tn;
    const uint32_t P = static_cast<uint32_t>(p.P);
    uint32_t c0, c1, CH;
    slice_chunks<BN>(p, sub, nsub, c0, c1, CH);
    const uint32_t set_bytes = CH * P;
    const uint32_t NB = min(3u, st.ring_bytes / set_bytes);
    const uint32_t nch = c1 - c0;   // chunks of this slice
    const char *src0 = partial_tile_at<BN>(p, 0, lt) + static_cast<size_t>(c0) * CH;
    const size_t rank_stride = static_cast<size_t>(p.num_tiles) * partial_tile_bytes<BN>(p);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](uint32_t ch, uint32_t seq) {
        const uint32_t b = seq % NB;
        const uint32_t bar = smem_u32(&st.rfull[b]);
        mbar_arrive_expect_tx(bar, set_bytes);
        for (uint32_t r = 0; r < P; ++r)
            bulk_load_evict_first(smem_u32(st.ring + b * set_bytes + r * CH), src0 + r * rank_stride + ch * CH, CH,
                                  bar, pol);
    };
    if (etid == 0)
        for (uint32_t k = 0; k < NB && k < nch; ++k) issue(k, st.seq + k);
    const int row = etid & (MK_BM - 1);
    const int half = etid >> 7;
    const int grow = tm * MK_BM + row;
    const uint32_t groups_per_chunk = CH / (MK_BM * 16);   // 4 (8 KiB) or 2 (4 KiB)
    for (uint32_t ch = 0; ch < nch; ++ch) {
        const uint32_t seq = st.seq + ch;
        const uint32_t b = seq % NB;
        wait_bar<false>(smem_u32(&st.rfull[b]), (seq / NB) & 1u, c, SITE_STAGE_FULL, ch);
        const uint8_t *buf = st.ring + b * set_bytes;
        if (p.partial_bf16) {
            // eight bf16 columns per 16-byte group, widened exactly to fp32 and summed in rank order
            const int ng = groups_per_chunk == 4 ? 2 : 1;
            const int g_local = groups_per_chunk == 4 ? 2 * half : half;
#pragma unroll 1
            for (int gi = 0; gi < ng; ++gi) {
                const uint32_t off = (static_cast<uint32_t>(g_local + gi) * MK_BM + row) * 16;
                float4 lo, hi;
                widen_bf16x8(*reinterpret_cast<const uint4 *>(buf + off), lo, hi);
                for (uint32_t r = 1; r < P; ++r) {
                    float4 xl, xh;
                    widen_bf16x8(*reinterpret_cast<const uint4 *>(buf + r * CH + off), xl, xh);
                    lo.x += xl.x; lo.y += xl.y; lo.z += xl.z; lo.w += xl.w;
                    hi.x += xh.x; hi.y += xh.y; hi.z += xh.z; hi.w += xh.w;
                }
                const int gcol = tn * BN + static_cast<int>((c0 + ch) * groups_per_chunk + g_local + gi) * 8;
                if (grow < p.M && gcol < p.N) store_out8(p, grow, gcol, lo, hi);
            }
        } else if (groups_per_chunk == 4) {
            const int g_local = 2 * half;   // this thread's two column groups in the chunk
            const uint32_t off0 = (static_cast<uint32_t>(g_local) * MK_BM + row) * 16;
            const uint32_t off1 = off0 + MK_BM * 16;
            float4 a0 = *reinterpret_cast<const float4 *>(buf + off0);
            float4 a1 = *reinterpret_cast<const float4 *>(buf + off1);
            for (uint32_t r = 1; r < P; ++r) {
                const float4 x0 = *reinterpret_cast<const float4 *>(buf + r * CH + off0);
                const float4 x1 = *reinterpret_cast<const float4 *>(buf + r * CH + off1);
                a0.x += x0.x; a0.y += x0.y; a0.z += x0.z; a0.w += x0.w;
                a1.x += x1.x; a1.y += x1.y; a1.z += x1.z; a1.w += x1.w;
            }
            const int gcol = tn * BN + static_cast<int>((c0 + ch) * 4 + g_local) * 4;
            if (grow < p.M && gcol < p.N) store_out8(p, grow, gcol, a0, a1);
        } else {
            const uint32_t off = (static_cast<uint32_t>(half) * MK_BM + row) * 16;
            float4 a = *reinterpret_cast<const float4 *>(buf + off);
            for (uint32_t r = 1; r < P; ++r) {
                const float4 x = *reinterpret_cast<const float4 *>(buf + r * CH + off);
                a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
            }
            const int gcol = tn * BN + static_cast<int>((c0 + ch) * 2 + half) * 4;
            if (grow < p.M && gcol < p.N) store_out4(p, grow, gcol, a);
        }
        bar_sync(1, MK_EPI_THREADS);   // every thread is done with buffer b
        if (etid == 0 && ch + NB < nch) {
            fence_proxy_async_smem();
            issue(ch + NB, seq + NB);
        }
    }
    st.seq += nch;
    if (etid == 0) fence_proxy_async_smem();   // the ring goes back to TMA loads after this item
}

// The reduce group (warps 2-9) handles one reduce item: slice sub of nsub of tile (tm, tn).
template <int BN>
__device__ void do_reduce(const MkParams &p, const Ctx &c, int tm, int tn, int sub, int nsub, int etid,
                          uint32_t epoch, Staging &st) {
    bool ok = true;
    const bool exists = tm < p.tiles_m;
    const int lt = tm * p.tiles_n + tn;
    if (exists && etid < 32) ok = wait_tile_ready(p, c, lt, epoch, etid);
    // The barrier orders every lane's flag acquire before what thread 0 does next; thread 0 then
    // orders those acquires (generic proxy) before its bulk copies of the partials (async proxy).
    ok = bar_and(1, MK_EPI_THREADS, ok);
    if (exists && ok && etid == 0) fence_proxy_async_global();
    if (exists && ok) {
        const long long t0 = clock64();
        reduce_tile_staged<BN>(p, c, tm, tn, sub, nsub, etid, st);
        if (p.discard) discard_tile<BN>(p, lt, sub, nsub, etid, MK_EPI_THREADS);
        if (etid == 0)
            atomicAdd(reinterpret_cast<unsigned long long *>(&c.hdr->reduce_busy),
                      static_cast<unsigned long long>(clock64() - t0));
    }
    if (etid == 0 && (ok || !exists)) atomicAdd(&c.hdr->tiles_done, 1u);
}

// Between the 32-column chunks of an epilogue's global stores: a pause, so that the 8 warps'
// stores do not arrive in one burst that holds up the TMA loads feeding the next unit (measured:
// up to 9 % faster GEMM at K_r = 1024).  The host sizes it to fit well inside one unit's MMA time.
__device__ __forceinline__ void epilogue_pace(const MkParams &p) {
    if (p.epi_pace_ns > 0) __nanosleep(static_cast<unsigned>(p.epi_pace_ns));
}

// The epilogue group drains TMEM accumulator `acc` (128 lanes x BN columns of fp32) into the
// partial tile (r, lt) with 512-byte coalesced warp stores.
template <int BN>
__device__ __forceinline__ void store_partial(const MkParams &p, uint32_t tmem_acc, int r, int lt, int warp,
                                              int lane) {
    const int lq = warp & 3;                          // the TMEM lane quarter this warp can access
    const int half = (warp - MK_EPI_WARP0) >> 2;      // which half of the tile's columns
    const int row = lq * 32 + lane;
    char *tile = partial_tile_at<BN>(p, r, lt);
    // partial tiles should live in L2 until the reduce role has read them (then they are
    // discarded); in rank-major order only the last rank's tiles are read soon after they are
    // written, the others would only crowd out the band's A rows
    const uint64_t pol = !p.l2_hints ? policy_evict_normal()
                         : (p.rank_major && r < p.P - 1) ? policy_evict_first() : policy_evict_last();
#pragma unroll 1
    for (int cc = 0; cc < BN / 64; ++cc) {
        const int col0 = half * (BN / 2) + cc * 32;
        uint32_t v[32];
        if (p.num_kb > 0) {
            tmem_ld32(tmem_acc + (static_cast<uint32_t>(lq * 32) << 16) + static_cast<uint32_t>(col0), v);
        } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = 0u;
        }
        if (p.partial_bf16) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                char *dst = tile + (static_cast<size_t>((col0 >> 3) + q) * MK_BM + row) * 16;
                st_u4_hint(dst, pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                           pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                           pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                           pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])), pol);
            }
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                char *dst = tile + (static_cast<size_t>((col0 >> 2) + q) * MK_BM + row) * 16;
                st_f4_hint(dst, __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]), pol);
            }
        }
        epilogue_pace(p);
    }
}

// ------------------------------------------------------------------ accumulate mode
// The ReduceScatter design the pages give for one node (Table 3, "GEMM + ReduceScatter"): the
// compute blocks themselves add each partial tile into the owner's fp32 buffer, here one fp32
// accumulator tile per output tile in the workspace (laid out like a partial tile), with L2
// reductions (red.add.v4.f32), so no partial tile is stored and read back and no reduce role
// exists.  The order in which the P ranks' additions land is not fixed, so results are exact
// for integer inputs and within rounding otherwise.  The block whose addition is the P-th
// (atomic count per tile, acquire-release) converts the tile to the output and clears the
// accumulator and the count for the next call.
template <int BN>
__device__ __forceinline__ void accumulate_partial(const MkParams &p, uint32_t tmem_acc, int lt, int r, int warp,
                                                   int lane) {
    const int lq = warp & 3;
    const int half = (warp - MK_EPI_WARP0) >> 2;
    const int row = lq * 32 + lane;
    float *tile = p.partials + static_cast<size_t>(lt) * (MK_BM * BN);
    const uint64_t pol = p.l2_hints ? policy_evict_last() : policy_evict_normal();
    // ranks of one tile often run at the same time: each starts on a different 32-column chunk,
    // so that their additions to the same lines do not all arrive together
#pragma unroll 1
    for (int i = 0; i < BN / 64; ++i) {
        const int cc = (i + r) % (BN / 64);
        const int col0 = half * (BN / 2) + cc * 32;
        uint32_t v[32];
        if (p.num_kb == 0) break;   // nothing to add
        tmem_ld32(tmem_acc + (static_cast<uint32_t>(lq * 32) << 16) + static_cast<uint32_t>(col0), v);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float *dst = tile + (static_cast<size_t>((col0 >> 2) + q) * MK_BM + row) * 4;
            red_add_f4_hint(dst, __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                            __uint_as_float(v[4 * q + 3]), pol);
        }
        epilogue_pace(p);
    }
}

// After every epilogue thread has issued its additions for tile (tm, tn): count this rank's
// contribution; the last contributor writes the tile's output and clears its accumulator.
template <int BN>
__device__ void finish_accumulate(const MkParams &p, const Ctx &c, int tm, int tn, int etid) {
    const int lt = tm * p.tiles_n + tn;
    bar_sync(1, MK_EPI_THREADS);   // all additions of this block issued (ordered before the release below)
    bool last = false;
    if (etid == 0) {
        __threadfence();
        last = atom_add_acq_rel_gpu(p.flags + lt, 1u) == static_cast<uint32_t>(p.P - 1);
    }
    last = bar_or(1, MK_EPI_THREADS, last);
    if (!last) return;
    __threadfence();
    const int row = etid & (MK_BM - 1);
    const int half = etid >> 7;
    const int grow = tm * MK_BM + row;
    float *tile = p.partials + static_cast<size_t>(lt) * (MK_BM * BN);
#pragma unroll 2
    for (int u = 0; u < BN / 16; ++u) {
        const int g0 = 4 * u + 2 * half;
        float4 *q0 = reinterpret_cast<float4 *>(tile) + static_cast<size_t>(g0) * MK_BM + row;
        const float4 a = ld_cg_f4(q0), b = ld_cg_f4(q0 + MK_BM);
        const int gcol = tn * BN + g0 * 4;
        if (grow < p.M && gcol < p.N) store_out8(p, grow, gcol, a, b);
        st_f4(q0, 0.f, 0.f, 0.f, 0.f);
        st_f4(q0 + MK_BM, 0.f, 0.f, 0.f, 0.f);
    }
    bar_sync(1, MK_EPI_THREADS);
    if (etid == 0) {
        st_relaxed_gpu(p.flags + lt, 0u);
        atomicAdd(&c.hdr->tiles_done, 1u);
    }
}

// ------------------------------------------------------------------ chained mode
// The rank-ordered sum built by the compute blocks themselves: the epilogue of unit (tile, r)
// waits for flag[tile][r-1] (rank r-1 has folded its partial in), adds its accumulator to the
// running sum S = ((p_0 + p_1) + ...) + p_{r-1} held in rank 0's partial tile, and stores the
// new sum, or for r = P-1 writes the output.  The fp32 additions are the ones the reduce role
// makes, in the same order, so the result is the same bit for bit; no reduce role is needed and
// a partial tile is read back only as the running sum, which the rank-major bands keep in L2.
// False if the wait for the predecessor gave up (the grid is aborting).
// Collective over the epilogue group: wait until rank r-1 has released the running sum of tile
// lt (nothing to wait for at r = 0).  False if the wait gave up (the grid is aborting).
__device__ bool wait_predecessor(const MkParams &p, const Ctx &c, int lt, int r, int lane, int etid, uint32_t epoch) {
    bool ok = true;
    if (r > 0 && etid < 32) {
        // lane 0 acquires the predecessor's flag (one flag: no need for the whole warp)
        const uint32_t *f = p.flags + static_cast<size_t>(lt) * p.P + (r - 1);
        int stop = 0;
        if (lane == 0) {
            uint64_t t0 = 0;
            for (uint32_t polls = 0; ld_acquire_gpu(f) != epoch; ++polls) {
                if (*c.s_abort) { stop = 1; break; }
                if (t0 == 0) t0 = globaltimer();
                if ((polls & 15u) == 15u) {
                    if (global_abort(c)) { stop = 1; break; }
                    if (globaltimer() - t0 > c.timeout_ns || polls > (1u << 30)) {
                        raise_error(c, MK_ERR_TIMEOUT, SITE_FLAG, static_cast<uint32_t>(lt * p.P + r - 1));
                        stop = 1;
                        break;
                    }
                }
                __nanosleep(32);
            }
        }
        ok = __shfl_sync(0xFFFFFFFFu, stop, 0) == 0;
    }
    return bar_and(1, MK_EPI_THREADS, ok);   // orders every thread's loads of S after the acquire
}

template <int BN>
__device__ bool chain_partial(const MkParams &p, const Ctx &c, uint32_t tmem_acc, int r, int tm, int tn, int warp,
                              int lane, int etid, uint32_t epoch) {
    const int lt = tm * p.tiles_n + tn;
    if (!wait_predecessor(p, c, lt, r, lane, etid, epoch)) return false;
    const int lq = warp & 3;
    const int half = (warp - MK_EPI_WARP0) >> 2;
    const int row = lq * 32 + lane;
    const int grow = tm * MK_BM + row;
    const bool last = r == p.P - 1;
    float *S = partial_tile<BN>(p, 0, lt);
    const uint64_t pol = p.l2_hints ? policy_evict_last() : policy_evict_normal();
    // The running sum is private to this mode, so it has a layout of its own: [BN/8 column
    // groups][128 rows][8 floats], which a thread reads and writes with 32-byte accesses (half the
    // store instructions of 16-byte ones; measured 1-2 % faster, and the stores are what the fold
    // costs the GEMM).
#pragma unroll 1
    for (int cc = 0; cc < BN / 64; ++cc) {
        const int col0 = half * (BN / 2) + cc * 32;
        float *base = S + (static_cast<size_t>(col0 >> 3) * MK_BM + row) * 8;
        // the running sum's loads go out first, so that their L2 latency overlaps the TMEM load
        float sv[4][8];
        if (r > 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) ld_cg_f8(base + q * MK_BM * 8, sv[q]);
        }
        uint32_t v[32];
        if (p.num_kb > 0) {
            tmem_ld32(tmem_acc + (static_cast<uint32_t>(lq * 32) << 16) + static_cast<uint32_t>(col0), v);
        } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = 0u;
        }
        float x[4][8];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < 8; ++j)   // S_{r-1} + p_r (fp32 addition commutes bit for bit)
                x[q][j] = r > 0 ? sv[q][j] + __uint_as_float(v[8 * q + j]) : __uint_as_float(v[8 * q + j]);
        if (last) {
            if (grow < p.M) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int gcol = tn * BN + col0 + 8 * q;
                    if (gcol < p.N)
                        store_out8(p, grow, gcol, make_float4(x[q][0], x[q][1], x[q][2], x[q][3]),
                                   make_float4(x[q][4], x[q][5], x[q][6], x[q][7]));
                }
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) st_f8_hint(base + q * MK_BM * 8, x[q], pol);
        }
        epilogue_pace(p);
    }
    return true;
}

// ------------------------------------------------------------------ split controller
// The split controller (one thread of block 0).  It reads the progress counters every
// ctrl_period_ns and publishes the number of reduce-role units.  Moving one reduce item from the
// end of the call into the compute phase costs the GEMM the SM time a reducer spends on it
// (tau, measured: reduce-role SM time per item), while reducing it at the end, when every SM
// reduces and the reduction runs at memory speed, costs the whole grid item_bytes / bandwidth,
// i.e. S * item_bytes / bandwidth SM time (tau_tail, computed by the host).  So the controller
// adds a reduce-role unit while the measured tau is below 0.8 tau_tail (early reduction is the
// cheaper place for the work) and removes one while it is above tau_tail, waiting dwell_ns
// between changes so the measurement can follow.  It starts from one unit and may go down to
// none, which leaves the whole reduction to the end of the call.  Once the compute
// queue is empty every unit reduces regardless of the target (see claim_work), the shift toward
// communication near the end of the GEMM.  The pages state the controller's inputs (progress
// counters) and output (a target number of communication blocks) but not its rule; this rule
// is a reading of that intent.  In static mode the thread only records the trace.  The loop
// doubles as a watchdog: no progress for timeout_ns raises MK_ERR_TIMEOUT.
__device__ void run_controller(const MkParams &p, const Ctx &c, uint32_t num_units, uint32_t num_items_total,
                               uint32_t done_per_unit, int role_units, int sms_per_role) {
    MkWsHeader *h = c.hdr;
    const int S = role_units * sms_per_role;
    const bool adaptive = p.mode == MK_MODE_ADAPTIVE && p.op != MK_IOP_AG;
    int cur = p.mode == MK_MODE_ADAPTIVE ? p.init_nr : p.static_nr;
    if (adaptive) st_relaxed_gpu(&h->target_nr, static_cast<uint32_t>(cur) + 1u);   // 0 = unpublished
    const uint64_t start = globaltimer();
    const long long clk0 = clock64();
    uint64_t last_change = start, last_adjust = start;
    uint32_t last_u = 0, last_d = 0;
    mk_trace_record *trace = static_cast<mk_trace_record *>(p.trace);
    uint32_t nrec = 0;
    uint64_t busy_mark = 0;
    uint32_t items_mark = 0;
    double tau_ns = -1.0;                        // EWMA of reduce-role SM time per item
    const double tau_tail = static_cast<double>(p.ctrl_tail_ns);
    const uint64_t dwell_ns = 4000;
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        const uint32_t u = ld_relaxed_gpu(&h->units_done);
        const uint32_t d = ld_relaxed_gpu(&h->tiles_done);
        const uint64_t now = globaltimer();
        if (trace && nrec < p.trace_cap) {
            mk_trace_record rec;
            rec.t_ns = now - start;
            // once the compute queue is empty every role unit reduces whatever the target says
            const bool drained = ld_relaxed_gpu(&h->compute_next) >= num_units;
            rec.target = static_cast<uint32_t>((drained ? role_units : cur) * sms_per_role);
            rec.units_done = u / done_per_unit;
            rec.tiles_done = d;
            rec.num_blocks = static_cast<uint32_t>(S);
            rec.reserved = 0;
            trace[nrec++] = rec;
        }
        if (d >= num_items_total || global_abort(c)) break;
        if (u != last_u || d != last_d) {
            last_u = u;
            last_d = d;
            last_change = now;
        } else if (now - last_change > c.timeout_ns) {
            raise_error(c, MK_ERR_TIMEOUT, SITE_WATCHDOG, d);
            break;
        }
        if (adaptive && u / done_per_unit < num_units) {
            if (d >= items_mark + 4 && now > start + 1000) {
                const uint64_t busy = ld_relaxed_gpu64(&h->reduce_busy);
                const double cyc_per_ns = static_cast<double>(clock64() - clk0) / static_cast<double>(now - start);
                const double t = static_cast<double>(busy - busy_mark) / (d - items_mark) / cyc_per_ns;
                tau_ns = tau_ns < 0.0 ? t : 0.75 * tau_ns + 0.25 * t;
                busy_mark = busy;
                items_mark = d;
            }
            if (tau_ns > 0.0 && now - last_adjust > dwell_ns) {
                int nr = cur;
                if (tau_ns < 0.8 * tau_tail && nr < role_units - 1) ++nr;
                else if (tau_ns > tau_tail && nr > 0) --nr;
                if (nr != cur) {
                    cur = nr;
                    last_adjust = now;
                    st_relaxed_gpu(&h->target_nr, static_cast<uint32_t>(cur) + 1u);
                }
            }
        }
        // once every unit is computed only the end of the call is left to notice: poll faster
        __nanosleep(u / done_per_unit < num_units ? static_cast<unsigned>(p.ctrl_period_ns) : 200u);
    }
    h->trace_count = nrec;
}

// Last block out resets the per-call counters and records the epoch it used.
__device__ void finish_call(const MkParams &p, uint32_t epoch) {
    MkWsHeader *h = p.hdr;
    __threadfence();
    const uint32_t prev = atomicAdd(&h->done_ctas, 1u);
    if (prev == gridDim.x - 1) {
        __threadfence();
        const uint32_t tiles_done = ld_relaxed_gpu(&h->tiles_done);
        const bool aborted = ld_relaxed_gpu(&h->abort) != 0u;
        h->compute_next = 0;
        h->reduce_next = 0;
        h->units_done = 0;
        h->tiles_done = 0;
        h->target_nr = 0;
        h->reduce_busy = 0;
        // accumulate mode has no waits to run out: a tile whose P contributions did not all
        // arrive shows up here as a missing output tile
        bool complete = true;
        if (p.mode == MK_MODE_ACCUMULATE && !aborted && tiles_done != static_cast<uint32_t>(p.num_tiles)) {
            complete = false;
            if (atomicCAS(&h->status, 0u, static_cast<uint32_t>(MK_ERR_INTERNAL)) == 0u) {
                h->err_site = SITE_ACC_STATE;
                h->err_index = tiles_done;
            }
        }
        // the accumulator region holds zeros after an accumulate call that ran to the end; any
        // other call leaves partial tiles (or an unfinished sum) there
        h->acc_state = (p.mode == MK_MODE_ACCUMULATE && !aborted && complete) ? MK_ACC_CLEAN : MK_ACC_DIRTY;
        h->abort = 0;
        h->epoch = epoch;
        h->done_ctas = 0;
        __threadfence();
    }
}

template <int STAGES>
__device__ void init_barriers(SmemCtl<STAGES> &s, const MkParams &p, uint32_t full_count, uint32_t tempty_count,
                              uint32_t wempty_count) {
    for (int i = 0; i < STAGES; ++i) {
        mbar_init(smem_u32(&s.full[i]), full_count);
        mbar_init(smem_u32(&s.empty[i]), 1);
    }
    for (int i = 0; i < ACC; ++i) {
        mbar_init(smem_u32(&s.tfull[i]), 1);
        mbar_init(smem_u32(&s.tempty[i]), tempty_count);
    }
    for (int i = 0; i < WQ; ++i) {
        mbar_init(smem_u32(&s.wfull[i]), 1);
        mbar_init(smem_u32(&s.wempty[i]), wempty_count);
    }
    mbar_init(smem_u32(&s.drain), 1);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&s.rfull[i]), 1);
    fence_mbar_init();
    s.abort = 0;
    s.issued = 0;
    s.peer_issued = 0;
    s.epi_done = 0;
    uint32_t e = ld_relaxed_gpu(&p.hdr->epoch) + 1u;
    if (e == 0u) e = 1u;
    s.epoch = e;
    // an accumulate call needs a zeroed accumulator: refuse (no block does any work) when the
    // last call on this workspace left partial tiles or an unfinished sum there
    if (p.mode == MK_MODE_ACCUMULATE && ld_relaxed_gpu(&p.hdr->acc_state) == MK_ACC_DIRTY) {
        if (atomicCAS(&p.hdr->status, 0u, static_cast<uint32_t>(MK_ERR_INVALID_ARG)) == 0u)
            p.hdr->err_site = SITE_ACC_STATE;
        atomicExch(&p.hdr->abort, 1u);
        s.abort = 1;
    }
}

// ----------------------------------------------------------------- AllGather + GEMM helpers
// Copy item i -> (destination rank r, 256-row pair row y): band by band (raster_group pair rows),
// rank by rank inside a band, the order in which the rank-major compute reads the gathered rows,
// so that rank r's copy of a band is complete as soon as its own share of copies is.  Each CTA of
// the pair copies one 128-row chunk (2y + its rank in the pair) to rank r's gathered buffer.
__device__ __forceinline__ void ag_item(const MkParams &p, int i, int &r, int &y) {
    const int G = p.raster_group;
    const int b = i / (G * p.P);
    const int rem = i - b * G * p.P;
    const int gsize = min(G, p.pair_tiles_m - b * G);
    r = rem / gsize;
    y = b * G + (rem - r * gsize);
}

// Readiness flag of 128-row chunk `chunk` in rank r's gathered copy of A.
__device__ __forceinline__ uint32_t *ag_flag(const MkParams &p, int chunk, int r) {
    return p.flags + static_cast<size_t>(r) * (2 * p.pair_tiles_m) + chunk;
}

// Producer thread: acquire the flag of 128-row chunk `chunk` of rank r's gathered A (bounded),
// then order the acquire before the TMA (async-proxy) reads of that chunk.
__device__ bool wait_chunk_ready(const MkParams &p, const Ctx &c, int chunk, int r, uint32_t epoch) {
    const uint32_t *f = ag_flag(p, chunk, r);
    uint64_t t0 = 0;
    for (uint32_t polls = 0; ld_acquire_gpu(f) != epoch; ++polls) {
        if (t0 == 0) t0 = globaltimer();
        if ((polls & 15u) == 15u) {
            if (global_abort(c)) return false;
            if (globaltimer() - t0 > c.timeout_ns || polls > (1u << 30)) {
                raise_error(c, MK_ERR_TIMEOUT, SITE_FLAG, static_cast<uint32_t>(chunk));
                return false;
            }
        }
        __nanosleep(64);
    }
    fence_proxy_async_global();
    return true;
}

// Epilogue group: TMEM accumulator (128 rows x BN fp32) -> rows tm*128.., columns tn*BN.. of the
// row-major M x N output C_r, in eight-column pieces (N is a multiple of 8).
template <int BN>
__device__ __forceinline__ void store_output_tile(const MkParams &p, uint32_t tmem_acc, int r, int tm, int tn,
                                                  int warp, int lane) {
    const int lq = warp & 3;
    const int half = (warp - MK_EPI_WARP0) >> 2;
    const int row = lq * 32 + lane;
    const int grow = tm * MK_BM + row;
#pragma unroll 1
    for (int cc = 0; cc < BN / 64; ++cc) {
        const int col0 = half * (BN / 2) + cc * 32;
        uint32_t v[32];
        if (p.num_kb > 0) {
            tmem_ld32(tmem_acc + (static_cast<uint32_t>(lq * 32) << 16) + static_cast<uint32_t>(col0), v);
        } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = 0u;
        }
        if (grow >= p.M) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int gcol = tn * BN + col0 + 8 * q;
            if (gcol >= p.N) break;
            const size_t idx = static_cast<size_t>(grow) * p.N + gcol;
            const float *f = reinterpret_cast<const float *>(&v[8 * q]);
            if (p.out_bf16)
                st_u4(static_cast<uint16_t *>(p.out[r]) + idx, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
            else {
                st_f4(static_cast<float *>(p.out[r]) + idx, f[0], f[1], f[2], f[3]);
                st_f4(static_cast<float *>(p.out[r]) + idx + 4, f[4], f[5], f[6], f[7]);
            }
        }
    }
}

// Communication item of AllGather + GEMM: copy rows [chunk*128, chunk*128+128) of the
// concatenated shards into every rank's gathered buffer, then release the chunk flag.  One
// thread drives bulk copies through the block's TMA ring: global -> shared in pieces of up to
// 48 KiB (two pieces ahead), shared -> global to the P destinations as bulk groups.  The
// chunk's rows are contiguous in the gathered buffers and, within one shard, in the source.
__device__ void do_copy_chunk(const MkParams &p, const Ctx &c, int chunk, int dst, int etid, uint32_t epoch,
                              Staging &st) {
    if (etid == 0 && chunk < p.tiles_m) {
        constexpr uint32_t PIECE = 48u * 1024u;
        const size_t row_bytes = static_cast<size_t>(p.Kr) * 2;
        const int row_begin = chunk * MK_BM;
        const int row_end = min(p.M, row_begin + MK_BM);
        // pieces: walk shard segments, each cut into PIECE-sized slices
        struct Piece { const char *src; size_t dst_off; uint32_t bytes; };
        auto piece_at = [&](uint32_t k, Piece &pc) -> bool {
            uint32_t seen = 0;
            for (int row = row_begin; row < row_end;) {
                const int sh = row / p.rows_per_shard;
                const int seg_end = min(row_end, (sh + 1) * p.rows_per_shard);
                const size_t seg_bytes = static_cast<size_t>(seg_end - row) * row_bytes;
                const uint32_t np = static_cast<uint32_t>((seg_bytes + PIECE - 1) / PIECE);
                if (k < seen + np) {
                    const size_t off = static_cast<size_t>(k - seen) * PIECE;
                    pc.src = static_cast<const char *>(p.ag_src[sh]) +
                             static_cast<size_t>(row - sh * p.rows_per_shard) * row_bytes + off;
                    pc.dst_off = static_cast<size_t>(row) * row_bytes + off;
                    pc.bytes = static_cast<uint32_t>(seg_bytes - off < PIECE ? seg_bytes - off : PIECE);
                    return true;
                }
                seen += np;
                row = seg_end;
            }
            return false;
        };
        auto load = [&](uint32_t k, const Piece &pc) {
            const uint32_t b = (st.seq + k) & 3u;
            const uint32_t bar = smem_u32(&st.rfull[b]);
            mbar_arrive_expect_tx(bar, pc.bytes);
            bulk_load(smem_u32(st.ring + b * PIECE), pc.src, pc.bytes, bar);
        };
        Piece pc[2];
        uint32_t k = 0;
        bool have0 = piece_at(0, pc[0]);
        bool have1 = have0 && piece_at(1, pc[1]);
        if (have0) load(0, pc[0]);
        if (have1) load(1, pc[1]);
        while (have0) {
            const uint32_t b = (st.seq + k) & 3u;
            wait_bar<false>(smem_u32(&st.rfull[b]), ((st.seq + k) >> 2) & 1u, c, SITE_STAGE_FULL, k);
            bulk_store(static_cast<char *>(p.ag_dst[dst]) + pc[0].dst_off, smem_u32(st.ring + b * PIECE), pc[0].bytes);
            bulk_commit();
            Piece next2;
            const bool have2 = have1 && piece_at(k + 2, next2);
            if (have2) {
                bulk_wait_read<2>();   // piece k - 2, the last user of buffer (k + 2) & 3, has been read
                load(k + 2, next2);
            }
            pc[0] = pc[1];
            pc[1] = next2;
            have0 = have1;
            have1 = have2;
            ++k;
        }
        bulk_wait_all();
        fence_proxy_async_global();
        st_release_gpu(ag_flag(p, chunk, dst), epoch);
        st.seq += k;
    }
    bar_sync(1, MK_EPI_THREADS);
    if (etid == 0) atomicAdd(&c.hdr->tiles_done, 1u);
}

// Producer side of the ring hand-over: a reduce item borrows the TMA ring for staging, so after
// queueing one the producer issues no further loads until the epilogue group has finished it.
__device__ bool wait_epilogue_done(const volatile uint32_t *epi_done, uint32_t count, const Ctx &c) {
    if (*epi_done >= count) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1; i != 0u; ++i) {
        if (*epi_done >= count) return true;
        if ((i & 63u) == 0u) {
            if (global_abort(c)) return false;   // the epilogue stops on an abort
            if (globaltimer() - t0 > c.pipe_timeout_ns) break;
        }
        __nanosleep(64);
    }
    raise_error(c, MK_ERR_TIMEOUT, SITE_STAGE_EMPTY, count);
    return false;
}

// ======================================================================= one-SM tiles
template <int BN>
__device__ void run1_producer(const MkParams &p, SmemCtl<Cfg1<BN>::STAGES> &s, uint8_t *stages, const Ctx &c) {
    using T = Cfg1<BN>;
    const ClaimGeom g{static_cast<uint32_t>(p.num_units), static_cast<uint32_t>(p.num_tiles * p.red_split),
                      blockIdx.x, gridDim.x, 1u, static_cast<uint32_t>(p.red_split), p.tiles_m};
    int stage = 0, wq = 0;
    uint32_t phase = 0, wphase = 0;
    bool exhausted = false, stop = false;
    // A rows are reused by every column of the raster group: keep them; B columns stream.
    const uint64_t pol_a = p.op_hints ? policy_evict_last() : policy_evict_normal();
    const uint64_t pol_b = p.op_hints ? policy_evict_first() : policy_evict_normal();
    uint32_t pushed = 0, ring_free_at = 0;   // ring free once the epilogue has finished ring_free_at items
    bool last_reduce = false;
    uint32_t target = 0;                     // adaptive split: target_nr as last read
    const bool ahead_mode = claims_ahead(p);
    uint32_t ahead = NO_CLAIM;               // compute unit claimed ahead, not yet queued
    while (!stop) {
        // Reduce items are claimed at most one ahead of the one in progress, so that the last
        // items of a call spread over the grid instead of queueing behind a few blocks.
        if (last_reduce && !wait_epilogue_done(&s.epi_done, pushed - 1, c)) break;
        const int2 it = ahead != NO_CLAIM ? item_claimed_ahead(p, c, g, ahead, exhausted, target)
                                          : claim_work(p, c, g, exhausted, target);
        ahead = NO_CLAIM;
        last_reduce = it.x == ITEM_REDUCE;
        if (p.mode == MK_MODE_ADAPTIVE) target = ld_relaxed_gpu(&c.hdr->target_nr);   // used by the next claim
        if (!wait_bar<false>(smem_u32(&s.wempty[wq]), wphase ^ 1u, c, SITE_WORK_EMPTY, 0)) break;
        s.items[wq] = it;
        mbar_arrive(smem_u32(&s.wfull[wq]));
        ++pushed;
        if (it.x == ITEM_REDUCE) ring_free_at = pushed;
        if (++wq == WQ) {
            wq = 0;
            wphase ^= 1u;
        }
        if (it.x == ITEM_END) break;
        if (it.x != ITEM_COMPUTE) continue;
        if (ahead_mode) ahead = atomicAdd(&c.hdr->compute_next, 1u);   // consumed at the next claim
        const int u = it.y;
        int r, tm, tn;
        unit_coords(p, p.tiles_m, u, tm, tn, r);
        if (!wait_epilogue_done(&s.epi_done, ring_free_at, c)) break;
        for (int kb = 0; kb < p.num_kb; ++kb) {
            if (!wait_bar<false>(smem_u32(&s.empty[stage]), phase ^ 1u, c, SITE_STAGE_EMPTY, u)) {
                stop = true;
                break;
            }
            const uint32_t fb = smem_u32(&s.full[stage]);
            uint8_t *sa = stages + stage * T::STAGE_BYTES;
            uint8_t *sb = sa + T::A_BYTES;
            mbar_arrive_expect_tx(fb, T::STAGE_BYTES);
            tma_load_2d_hint(smem_u32(sa), &p.tmA[r], fb, kb * MK_BK, tm * MK_BM, pol_a);
            if (p.b_nk) {   // B given as N x K_r: the tile's BN rows of this K slice, one box
                tma_load_2d_hint(smem_u32(sb), &p.tmB[r], fb, kb * MK_BK, tn * BN, pol_b);
            } else {
#pragma unroll
                for (int j = 0; j < T::B_BOXES; ++j)
                    tma_load_2d_hint(smem_u32(sb + j * T::B_BOX_BYTES), &p.tmB[r], fb, tn * BN + j * 64,
                                     kb * MK_BK, pol_b);
            }
            ++s.issued;
            if (++stage == T::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    // Every TMA load this thread issued must have landed before the block exits (normally the
    // MMA warp has waited for all of them already; this matters after a pipeline timeout).
    const uint32_t n = s.issued;
    for (uint32_t i = n > T::STAGES ? n - T::STAGES : 0; i < n; ++i)
        wait_bar<false>(smem_u32(&s.full[i % T::STAGES]), (i / T::STAGES) & 1u, c, SITE_DRAIN, i);
}

template <int BN>
__device__ void run1_mma(const MkParams &p, SmemCtl<Cfg1<BN>::STAGES> &s, uint8_t *stages, const Ctx &c,
                         uint32_t tmem_base) {
    using T = Cfg1<BN>;
    const uint32_t b_lbo = p.b_nk ? 16u : static_cast<uint32_t>(T::B_BOX_BYTES);   // as in run2_mma
    const uint64_t b_kstep = p.b_nk ? 2u : 128u;
    const uint32_t idesc = p.b_nk ? (T::IDESC & ~(1u << 16)) : T::IDESC;
    int stage = 0, acc = 0, wq = 0;
    uint32_t phase = 0, aphase = 0, wphase = 0;
    for (;;) {
        if (!wait_bar<false>(smem_u32(&s.wfull[wq]), wphase, c, SITE_WORK_FULL, 0)) break;
        const int2 it = s.items[wq];
        mbar_arrive(smem_u32(&s.wempty[wq]));
        if (++wq == WQ) {
            wq = 0;
            wphase ^= 1u;
        }
        if (it.x == ITEM_END) break;
        if (it.x != ITEM_COMPUTE) continue;
        if (!wait_bar<false>(smem_u32(&s.tempty[acc]), aphase ^ 1u, c, SITE_ACC_EMPTY, it.y)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < p.num_kb; ++kb) {
            if (!wait_bar<false>(smem_u32(&s.full[stage]), phase, c, SITE_STAGE_FULL, it.y)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(stages + stage * T::STAGE_BYTES);
            const uint32_t sb = sa + T::A_BYTES;
            // A: K-major, rows 128 B apart, 8-row groups 1024 B apart; K step of 16 = +32 B.
            // B: MN-major, 64-column boxes 8 KiB apart (LBO), 8-row K groups 1024 B apart (SBO);
            //    K step of 16 rows = +2048 B.  With b_nk, B is K-major like A.
            const uint64_t ad = sw128_desc(sa, 16, 1024);
            const uint64_t bd = sw128_desc(sb, b_lbo, 1024);
#pragma unroll
            for (int kk = 0; kk < MK_BK / 16; ++kk)
                umma_bf16(d_tmem, ad + static_cast<uint64_t>(kk * 2), bd + static_cast<uint64_t>(kk) * b_kstep, idesc,
                          static_cast<uint32_t>((kb | kk) != 0));
            umma_commit(smem_u32(&s.empty[stage]));
            if (++stage == T::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        umma_commit(smem_u32(&s.tfull[acc]));
        if (++acc == ACC) {
            acc = 0;
            aphase ^= 1u;
        }
    }
    // Every MMA issued by this thread must complete before TMEM is released.
    umma_commit(smem_u32(&s.drain));
    wait_bar<false>(smem_u32(&s.drain), 0, c, SITE_DRAIN, 0);
}

template <int BN>
__device__ void run1_epilogue(const MkParams &p, SmemCtl<Cfg1<BN>::STAGES> &s, uint8_t *stages, const Ctx &c,
                              uint32_t tmem_base, uint32_t epoch) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int etid = threadIdx.x - MK_EPI_WARP0 * 32;
    Staging st{stages, Cfg1<BN>::STAGES * Cfg1<BN>::STAGE_BYTES, s.rfull, 0};
    int acc = 0, wq = 0;
    uint32_t aphase = 0, wphase = 0;
    for (;;) {
        bool ok = true;
        if (lane == 0) ok = wait_bar<false>(smem_u32(&s.wfull[wq]), wphase, c, SITE_WORK_FULL, 0);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!bar_and(1, MK_EPI_THREADS, ok)) break;
        const int2 it = s.items[wq];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.wempty[wq]));
        if (++wq == WQ) {
            wq = 0;
            wphase ^= 1u;
        }
        if (it.x == ITEM_END) break;
        if (it.x == ITEM_COMPUTE) {
            const int u = it.y;
            int r, tm, tn;
            unit_coords(p, p.tiles_m, u, tm, tn, r);
            const int lt = tm * p.tiles_n + tn;
            ok = true;
            if (lane == 0) ok = wait_bar<false>(smem_u32(&s.tfull[acc]), aphase, c, SITE_ACC_FULL, u);
            ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
            if (!bar_and(1, MK_EPI_THREADS, ok)) break;
            tc_fence_after();
            const bool accumulate = p.mode == MK_MODE_ACCUMULATE;
            const bool chained = p.mode == MK_MODE_CHAINED;
            bool folded = true;
            if (accumulate)
                accumulate_partial<BN>(p, tmem_base + static_cast<uint32_t>(acc * BN), lt, r, warp, lane);
            else if (chained)
                folded = chain_partial<BN>(p, c, tmem_base + static_cast<uint32_t>(acc * BN), r, tm, tn, warp, lane,
                                           etid, epoch);
            else
                store_partial<BN>(p, tmem_base + static_cast<uint32_t>(acc * BN), r, lt, warp, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.tempty[acc]));
            if (++acc == ACC) {
                acc = 0;
                aphase ^= 1u;
            }
            if (accumulate) {
                finish_accumulate<BN>(p, c, tm, tn, etid);
                if (etid == 0) atomicAdd(&c.hdr->units_done, 1u);
            } else {
                bar_sync(1, MK_EPI_THREADS);   // every store of this partial tile has been issued
                if (etid == 0 && folded) {
                    st_release_gpu(p.flags + static_cast<size_t>(lt) * p.P + r, epoch);
                    atomicAdd(&c.hdr->units_done, 1u);
                    if (chained && r == p.P - 1) atomicAdd(&c.hdr->tiles_done, 1u);
                }
            }
        } else {
            int tm, tn;
            raster(it.y / p.red_split, p.tiles_m, p.tiles_n, p.raster_group, tm, tn);
            do_reduce<BN>(p, c, tm, tn, it.y % p.red_split, p.red_split, etid, epoch, st);
        }
        if (etid == 0) *reinterpret_cast<volatile uint32_t *>(&s.epi_done) = s.epi_done + 1;
    }
}

template <int BN>
__global__ void __launch_bounds__(MK_THREADS, 1) mk_persistent_kernel(const __grid_constant__ MkParams p) {
    using T = Cfg1<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                  ~static_cast<uintptr_t>(1023));
    SmemCtl<T::STAGES> &s = *reinterpret_cast<SmemCtl<T::STAGES> *>(stages + T::STAGES * T::STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) init_barriers<T::STAGES>(s, p, 1, MK_EPI_THREADS / 32, 1 + MK_EPI_THREADS / 32);
    if (warp == 0 && lane == 0)
        for (int r = 0; r < p.P; ++r) {
            prefetch_tmap(&p.tmA[r]);
            prefetch_tmap(&p.tmB[r]);
        }
    if (warp == 1) {
        tmem_alloc(smem_u32(&s.tmem_base), T::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;
    const uint32_t epoch = s.epoch;
    const Ctx c{p.hdr, &s.abort, p.timeout_ns, 4 * p.timeout_ns};

    if (warp == 0) {
        if (lane == 0) run1_producer<BN>(p, s, stages, c);
    } else if (warp == 1) {
        if (lane == 0) run1_mma<BN>(p, s, stages, c, tmem_base);
    } else if (warp < MK_CTRL_WARP) {
        run1_epilogue<BN>(p, s, stages, c, tmem_base, epoch);
    } else if (lane == 0 && blockIdx.x == 0 &&
               (p.mode == MK_MODE_ADAPTIVE || (p.mode == MK_MODE_STATIC && p.trace))) {
        run_controller(p, c, p.num_units, p.num_tiles * p.red_split, 1, gridDim.x, 1);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, T::TMEM_COLS);
    if (threadIdx.x == 0) finish_call(p, epoch);
}

// ======================================================================= SM-pair tiles
// Pair geometry: pair tile (sm, tn) covers tile rows 2*sm (even CTA) and 2*sm+1 (odd CTA).
// Compute unit u = pair_tile * P + r; reduce item i = pair tile i (each CTA reduces its row).
//
// Barriers (same offsets in both CTAs; the even CTA's copy is the one used where noted):
//   full[s]   even CTA, 2 arrivals (both producers' expect_tx) + both CTAs' TMA bytes
//   empty[s]  both, 1 arrival: the MMA commit multicast to both CTAs
//   tfull[a]  both, 1 arrival: commit multicast
//   tempty[a] even CTA, 16 arrivals: 8 epilogue warps of each CTA
//   wfull[q]  both, 1 arrival: the even CTA's scheduler
//   wempty[q] even CTA, 18 arrivals: MMA + 8 epilogue warps (even), producer + 8 epilogue (odd)
template <int BN>
__device__ void run2_producer(const MkParams &p, SmemCtl<Cfg2<BN>::STAGES> &s, uint8_t *stages, const Ctx &c,
                              uint32_t crank) {
    using T = Cfg2<BN>;
    const bool leader = crank == 0;
    const bool ag = p.op == MK_IOP_AG;
    // tile owners (chained mode, short M) claim whole tiles and load the tile's P ranks in turn
    const ClaimGeom g{static_cast<uint32_t>((BN == 128 && p.chain_owner) ? p.num_pair_tiles : p.num_pair_units),
                      static_cast<uint32_t>(ag ? p.P * p.pair_tiles_m : p.num_pair_tiles * p.red_split), blockIdx.x >> 1,
                      gridDim.x >> 1, 2u, ag ? 1u : static_cast<uint32_t>(p.red_split), p.pair_tiles_m};
    const uint32_t full0 = mapa_shared(smem_u32(&s.full[0]), 0);      // even CTA's full barriers
    const uint32_t wempty0 = mapa_shared(smem_u32(&s.wempty[0]), 0);
    const uint32_t peer_items = mapa_shared(smem_u32(&s.items[0]), 1);
    const uint32_t peer_wfull = mapa_shared(smem_u32(&s.wfull[0]), 1);
    int stage = 0, wq = 0;
    uint32_t phase = 0, wphase = 0;
    bool exhausted = false, stop = false;
    const uint64_t pol_a = p.op_hints ? policy_evict_last() : policy_evict_normal();
    const uint64_t pol_b = p.op_hints ? policy_evict_first() : policy_evict_normal();
    uint32_t pushed = 0, ring_free_at = 0;
    bool last_reduce = false;
    uint32_t target = 0;   // adaptive split: target_nr as last read (see claim_work)
    const bool ahead_mode = leader && claims_ahead(p);
    uint32_t ahead = NO_CLAIM;   // compute unit claimed ahead, not yet queued
    while (!stop) {
        int2 it;
        if (leader) {
            // reduce items: at most one claimed ahead of the one in progress (see run1_producer)
            if (last_reduce && !wait_epilogue_done(&s.epi_done, pushed - 1, c)) break;
            it = ahead != NO_CLAIM ? item_claimed_ahead(p, c, g, ahead, exhausted, target)
                                   : claim_work(p, c, g, exhausted, target);
            ahead = NO_CLAIM;
            last_reduce = it.x == ITEM_REDUCE;
            if (p.mode == MK_MODE_ADAPTIVE) target = ld_relaxed_gpu(&c.hdr->target_nr);   // used by the next claim
            if (!wait_bar<true>(smem_u32(&s.wempty[wq]), wphase ^ 1u, c, SITE_WORK_EMPTY, 0)) break;
            s.items[wq] = it;
            st_cluster_v2(peer_items + 8u * wq, it.x, it.y);
            mbar_arrive(smem_u32(&s.wfull[wq]));
            mbar_arrive_cluster(peer_wfull + 8u * wq);
        } else {
            if (!wait_bar<true>(smem_u32(&s.wfull[wq]), wphase, c, SITE_WORK_FULL, 0)) break;
            it = s.items[wq];
            mbar_arrive_cluster(wempty0 + 8u * wq);
        }
        if (++wq == WQ) {
            wq = 0;
            wphase ^= 1u;
        }
        ++pushed;
        if (it.x == ITEM_REDUCE) ring_free_at = pushed;
        if (it.x == ITEM_END) break;
        if (it.x != ITEM_COMPUTE) continue;
        if (ahead_mode) ahead = atomicAdd(&c.hdr->compute_next, 1u);   // consumed at the next claim
        const int u = it.y;
        if (!wait_epilogue_done(&s.epi_done, ring_free_at, c)) break;
        // a unit's ranks (chained mode: chain_ranks of them; otherwise one), or a tile owner's P
        // ranks (tile owners exist only with 128-column tiles)
        const bool owner = BN == 128 && p.chain_owner;
        int sm, tn, r0 = 0, nranks = p.P;
        if (owner)
            raster(u, p.pair_tiles_m, p.tiles_n, p.raster_group, sm, tn);
        else
            unit_span(p, u, sm, tn, r0, nranks);
        for (int rr = 0; rr < nranks && !stop; ++rr) {
            const int r = r0 + rr;
            const int tm = 2 * sm + static_cast<int>(crank);
            const CUtensorMap *amap = &p.tmA[r];
            int ay = tm * MK_BM;
            if (p.op == MK_IOP_AG) {
                if (p.ag_gather) {
                    // a failed wait has raised the abort: the loads still go ahead so the pipeline drains
                    if (p.ag_wait && tm < p.tiles_m) (void)wait_chunk_ready(p, c, tm, r, s.epoch);
                } else {
                    const int sh = min(p.P - 1, tm * MK_BM / p.rows_per_shard);   // rows_per_shard % 128 == 0
                    amap = &p.tmA[sh];
                    ay = tm * MK_BM - sh * p.rows_per_shard;
                }
            }
            for (int kb = 0; kb < p.num_kb; ++kb) {
                if (!wait_bar<false>(smem_u32(&s.empty[stage]), phase ^ 1u, c, SITE_STAGE_EMPTY, u)) {
                    stop = true;
                    break;
                }
                const uint32_t fb = full0 + 8u * stage;
                const uint32_t sa = smem_u32(stages + stage * T::STAGE_BYTES);
                const uint32_t sb = sa + T::A_BYTES;
                mbar_arrive_expect_tx_cluster(fb, T::STAGE_BYTES);
                tma_load_2d_pair_hint(sa, amap, fb, kb * MK_BK, ay, pol_a);
                if (p.b_nk) {   // B given as N x K_r: this CTA's BN/2 rows of the K slice, one box
                    tma_load_2d_pair_hint(sb, &p.tmB[r], fb, kb * MK_BK, tn * BN + static_cast<int>(crank) * (BN / 2),
                                          pol_b);
                } else {
#pragma unroll
                    for (int j = 0; j < T::B_BOXES; ++j)
                        tma_load_2d_pair_hint(sb + j * T::B_BOX_BYTES, &p.tmB[r], fb,
                                              tn * BN + static_cast<int>(crank) * (BN / 2) + j * 64, kb * MK_BK, pol_b);
                }
                ++s.issued;
                if (++stage == T::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
    // The even CTA's MMA commits arrive (multicast) on this CTA's empty barriers once the MMAs
    // that read each stage complete.  Wait for the arrivals that free the last stages this
    // producer filled, so that no such arrive is still in flight when the CTA exits.
    const uint32_t n = s.issued;
    for (uint32_t i = n > T::STAGES ? n - T::STAGES : 0; i < n; ++i)
        wait_bar<false>(smem_u32(&s.empty[i % T::STAGES]), (i / T::STAGES) & 1u, c, SITE_DRAIN, i);
}

template <int BN>
__device__ void run2_mma(const MkParams &p, SmemCtl<Cfg2<BN>::STAGES> &s, uint8_t *stages, const Ctx &c,
                         uint32_t tmem_base) {
    using T = Cfg2<BN>;
    // B operand: MN-major 64-column boxes (K x N input; K advances by 16 rows = 2 KiB), or K-major
    // rows like A (N x K input; K advances by 16 elements = 32 bytes), descriptor units of 16 bytes
    const uint32_t b_lbo = p.b_nk ? 16u : static_cast<uint32_t>(T::B_BOX_BYTES);
    const uint64_t b_kstep = p.b_nk ? 2u : 128u;
    const uint32_t idesc = p.b_nk ? (T::IDESC & ~(1u << 16)) : T::IDESC;
    int stage = 0, acc = 0, wq = 0;
    uint32_t phase = 0, aphase = 0, wphase = 0;
    for (;;) {
        if (!wait_bar<true>(smem_u32(&s.wfull[wq]), wphase, c, SITE_WORK_FULL, 0)) break;
        const int2 it = s.items[wq];
        mbar_arrive(smem_u32(&s.wempty[wq]));
        if (++wq == WQ) {
            wq = 0;
            wphase ^= 1u;
        }
        if (it.x == ITEM_END) break;
        if (it.x != ITEM_COMPUTE) continue;
        // one unit's ranks (one, or two with chain_ranks = 2), or a tile owner's P ranks, each in
        // the next accumulator (tile owners exist only with 128-column tiles)
        int nranks = 1;
        if (BN == 128 && p.chain_owner) {
            nranks = p.P;
        } else if (p.chain_ranks > 1) {
            int sm, tn, r0;
            unit_span(p, it.y, sm, tn, r0, nranks);
        }
        bool ok = true;
        for (int rr = 0; rr < nranks && ok; ++rr) {
            if (!wait_bar<false>(smem_u32(&s.tempty[acc]), aphase ^ 1u, c, SITE_ACC_EMPTY, it.y)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
            for (int kb = 0; kb < p.num_kb; ++kb) {
                if (!wait_bar<false>(smem_u32(&s.full[stage]), phase, c, SITE_STAGE_FULL, it.y)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(stages + stage * T::STAGE_BYTES);
                const uint32_t sb = sa + T::A_BYTES;
                // Per-CTA halves at identical offsets in both CTAs: A 128 rows (K-major), B BN/2
                // columns (MN-major, 64-column boxes 8 KiB apart).
                const uint64_t ad = sw128_desc(sa, 16, 1024);
                const uint64_t bd = sw128_desc(sb, b_lbo, 1024);
#pragma unroll
                for (int kk = 0; kk < MK_BK / 16; ++kk)
                    umma_bf16_pair(d_tmem, ad + static_cast<uint64_t>(kk * 2), bd + static_cast<uint64_t>(kk) * b_kstep,
                                   idesc, static_cast<uint32_t>((kb | kk) != 0));
                umma_commit_pair(smem_u32(&s.empty[stage]), 0x3);
                if (++stage == T::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit_pair(smem_u32(&s.tfull[acc]), 0x3);
            if (++acc == ACC) {
                acc = 0;
                aphase ^= 1u;
            }
        }
        if (!ok) break;
    }
    umma_commit_pair(smem_u32(&s.drain), 0x1);
    wait_bar<false>(smem_u32(&s.drain), 0, c, SITE_DRAIN, 0);
}

// Tile owner (chained mode on a short M): the pair computed the P ranks of one 256 x 128 tile
// into alternating accumulators; the epilogue folds them, in rank order, into a running sum
// S = ((p_0 + p_1) + ...) + p_r kept in TMEM next to the accumulators (each thread its row's 64
// columns of the CTA's 128-row half), then writes the output once.  These are the reduce role's fp32
// additions in its order, so the bits are the same; nothing is stored before the output and no
// wait depends on another block.  False if a wait gave up (the grid is aborting).
template <int BN>
__device__ bool owner_tile(const MkParams &p, SmemCtl<Cfg2<BN>::STAGES> &s, const Ctx &c, uint32_t tmem_base, int pt,
                           uint32_t crank, int warp, int lane, int etid, int &acc, uint32_t &aphase,
                           uint32_t tempty0) {
    if constexpr (BN != 128) {
        // the host picks tile owners with 128-column tiles only
        if (etid == 0) raise_error(c, MK_ERR_INTERNAL, SITE_ACC_FULL, static_cast<uint32_t>(pt));
        return false;
    } else {
        int sm, tn;
        raster(pt, p.pair_tiles_m, p.tiles_n, p.raster_group, sm, tn);
        const int tm = 2 * sm + static_cast<int>(crank);
        const bool exists = tm < p.tiles_m;
        const int lq = warp & 3;
        const int half = (warp - MK_EPI_WARP0) >> 2;
        const int row = lq * 32 + lane;
        const int grow = tm * MK_BM + row;
        const uint32_t lanes = static_cast<uint32_t>(lq * 32) << 16;
        // the running sum lives in the TMEM columns after the two accumulators, in the same layout
        const uint32_t t_sum = tmem_base + static_cast<uint32_t>(ACC * BN) + lanes + static_cast<uint32_t>(half * 64);
#pragma unroll 1
        for (int r = 0; r < p.P; ++r) {
            bool ok = true;
            if (lane == 0) ok = wait_bar<false>(smem_u32(&s.tfull[acc]), aphase, c, SITE_ACC_FULL, pt);
            ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
            if (!bar_and(1, MK_EPI_THREADS, ok)) return false;
            tc_fence_after();
            if (exists) {
                const uint32_t t_acc = tmem_base + static_cast<uint32_t>(acc * BN) + lanes + static_cast<uint32_t>(half * 64);
                const bool last = r == p.P - 1;
#pragma unroll 1
                for (int h = 0; h < 4; ++h) {   // 16 of the thread's 64 columns at a time
                    uint32_t v[16], sv[16];
                    if (p.num_kb > 0) {
                        tmem_ld16(t_acc + static_cast<uint32_t>(16 * h), v);
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q) v[q] = 0u;
                    }
                    if (r > 0) {
                        tmem_ld16(t_sum + static_cast<uint32_t>(16 * h), sv);
#pragma unroll
                        for (int q = 0; q < 16; ++q)   // S_{r-1} + p_r (fp32 addition commutes bit for bit)
                            v[q] = __float_as_uint(__uint_as_float(sv[q]) + __uint_as_float(v[q]));
                    }
                    if (!last) {
                        tmem_st16(t_sum + static_cast<uint32_t>(16 * h), v);
                    } else if (grow < p.M) {
#pragma unroll
                        for (int g = 0; g < 2; ++g) {
                            const int gcol = tn * BN + half * 64 + 16 * h + 8 * g;
                            if (gcol < p.N)
                                store_out8(p, grow, gcol,
                                           make_float4(__uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1]),
                                                       __uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3])),
                                           make_float4(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]),
                                                       __uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7])));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (crank == 0) mbar_arrive(smem_u32(&s.tempty[acc]));
                else mbar_arrive_remote(tempty0 + 8u * acc);
            }
            if (++acc == ACC) {
                acc = 0;
                aphase ^= 1u;
            }
        }
        bar_sync(1, MK_EPI_THREADS);
        if (etid == 0) {
            atomicAdd(&c.hdr->units_done, static_cast<uint32_t>(p.P));
            if (exists) atomicAdd(&c.hdr->tiles_done, 1u);
        }
        return true;
    }
}

// Chained mode on SM pairs with several ranks per unit: ranks r0 .. r0 + nr - 1 of a tile land in
// the two TMEM accumulators in turn.  While the second rank's MMAs run, the epilogue adds the
// running sum S_{r0-1} (read once from L2, after rank r0-1's flag) to the first accumulator in
// place.  Each later accumulator, once complete, gets the sum so far added to it in place, and the
// accumulator that held the sum goes back to the MMA warp for the next rank.  The last sum is
// stored (the running sum for rank r0 + nr, or the output after rank P-1).  The additions are
// ((S_{r0-1} + p_r0) + p_{r0+1}) + ..., the reduce role's in its order, so the bits are the same,
// and the running sum crosses L2 once per nr ranks.  A unit with one rank folds like
// chain_partial.  False if a wait gave up (the grid is aborting).
template <int BN>
__device__ bool chain_span(const MkParams &p, SmemCtl<Cfg2<BN>::STAGES> &s, const Ctx &c, uint32_t tmem_base, int u,
                           uint32_t crank, int warp, int lane, int etid, int &acc, uint32_t &aphase, uint32_t tempty0,
                           uint32_t epoch) {
    int sm, tn, r0, nr;
    unit_span(p, u, sm, tn, r0, nr);
    const int tm = 2 * sm + static_cast<int>(crank);
    const bool exists = tm < p.tiles_m;
    const int lt = tm * p.tiles_n + tn;
    const bool last = r0 + nr == p.P;
    const bool kz = p.num_kb == 0;   // K_r = 0: the MMAs never wrote the accumulators, every p_r is 0
    const int lq = warp & 3;
    const int half = (warp - MK_EPI_WARP0) >> 2;
    const int row = lq * 32 + lane;
    const int grow = tm * MK_BM + row;
    const uint32_t lanes = static_cast<uint32_t>(lq * 32) << 16;
    auto wait_acc = [&]() -> bool {   // the accumulator `acc` is complete
        bool ok = true;
        if (lane == 0) ok = wait_bar<false>(smem_u32(&s.tfull[acc]), aphase, c, SITE_ACC_FULL, u);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!bar_and(1, MK_EPI_THREADS, ok)) return false;
        tc_fence_after();
        return true;
    };
    auto release = [&](int a) {   // hand accumulator `a` back to the MMA warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            if (crank == 0) mbar_arrive(smem_u32(&s.tempty[a]));
            else mbar_arrive_remote(tempty0 + 8u * a);
        }
    };
    auto next_acc = [&]() {
        if (++acc == ACC) {
            acc = 0;
            aphase ^= 1u;
        }
    };
    auto acc_ld = [&](uint32_t taddr, bool zero, uint32_t (&v)[16]) {
        if (zero) {
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = 0u;
        } else {
            tmem_ld16(taddr, v);
        }
    };
    if (!wait_acc()) return false;
    bool folded = true;
    if (nr == 1) {
        if (exists)
            folded = chain_partial<BN>(p, c, tmem_base + static_cast<uint32_t>(acc * BN), r0, tm, tn, warp, lane, etid,
                                       epoch);
        release(acc);
        next_acc();
    } else {
        float *S = partial_tile<BN>(p, 0, lt);
        // S_{r0-1} + p_r0 into the first accumulator (at r0 = 0, p_0 starts the sum as it is)
        if (exists && r0 > 0) {
            folded = wait_predecessor(p, c, lt, r0, lane, etid, epoch);
            if (folded) {
                const uint32_t ta = tmem_base + static_cast<uint32_t>(acc * BN) + lanes;
                // 32 of the thread's BN/2 columns at a time: the running sum's L2 loads for both
                // 16-column halves go out before the first is used, one round trip per 32 columns
#pragma unroll 1
                for (int cg = 0; cg < BN / 32; cg += 2) {
                    float sv[4][8];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int col0 = half * (BN / 2) + (cg + k) * 16;
                        const float *base = S + (static_cast<size_t>(col0 >> 3) * MK_BM + row) * 8;
                        ld_cg_f8(base, sv[2 * k]);
                        ld_cg_f8(base + MK_BM * 8, sv[2 * k + 1]);
                    }
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int col0 = half * (BN / 2) + (cg + k) * 16;
                        uint32_t v[16];
                        acc_ld(ta + static_cast<uint32_t>(col0), kz, v);
#pragma unroll
                        for (int q = 0; q < 2; ++q)
#pragma unroll
                            for (int j = 0; j < 8; ++j)   // fp32 addition commutes bit for bit
                                v[8 * q + j] = __float_as_uint(sv[2 * k + q][j] + __uint_as_float(v[8 * q + j]));
                        tmem_st16(ta + static_cast<uint32_t>(col0), v);
                    }
                }
            }
        }
        // the sum so far, in accumulator `acc`, into each later rank's accumulator (with K_r = 0
        // every p_r and so every sum is +0, and the accumulators hold nothing to read)
        for (int i = 1; i < nr; ++i) {
            const int prev = acc;
            next_acc();
            if (!wait_acc()) return false;
            if (exists && folded && !kz) {
                // the MMAs of the next rank wait for `prev`: the loads of 32 columns of both
                // accumulators go out together (one wait per 32 columns) and the stores are
                // waited for once, at the end
                const uint32_t ta = tmem_base + static_cast<uint32_t>(prev * BN) + lanes;
                const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * BN) + lanes;
#pragma unroll 1
                for (int cc = 0; cc < BN / 32; cc += 2) {   // 32 of the thread's BN/2 columns at a time
                    const uint32_t col0 = static_cast<uint32_t>(half * (BN / 2) + cc * 16);
                    uint32_t va[16], vb[16], vc[16], vd[16];
                    tmem_ld16_nowait(ta + col0, va);
                    tmem_ld16_nowait(tb + col0, vb);
                    tmem_ld16_nowait(ta + col0 + 16, vc);
                    tmem_ld16_nowait(tb + col0 + 16, vd);
                    tmem_wait_ld16(va);
                    tmem_wait_ld16(vb);
                    tmem_wait_ld16(vc);
                    tmem_wait_ld16(vd);
#pragma unroll
                    for (int q = 0; q < 16; ++q) vb[q] = __float_as_uint(__uint_as_float(va[q]) + __uint_as_float(vb[q]));
#pragma unroll
                    for (int q = 0; q < 16; ++q) vd[q] = __float_as_uint(__uint_as_float(vc[q]) + __uint_as_float(vd[q]));
                    tmem_st16_nowait(tb + col0, vb);
                    tmem_st16_nowait(tb + col0 + 16, vd);
                }
                tmem_wait_st();
            }
            release(prev);   // the next rank's MMAs may start in it
        }
        // the last accumulator out: the next running sum, or the output
        if (exists && folded) {
            const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * BN) + lanes;
            const uint64_t pol = p.l2_hints ? policy_evict_last() : policy_evict_normal();
#pragma unroll 1
            for (int cc = 0; cc < BN / 64; ++cc) {
                const int col0 = half * (BN / 2) + cc * 32;
                uint32_t v[32];
                if (kz) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] = 0u;
                } else {
                    tmem_ld32(tb + static_cast<uint32_t>(col0), v);
                }
                if (last) {
                    if (grow < p.M) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int gcol = tn * BN + col0 + 8 * q;
                            if (gcol < p.N)
                                store_out8(p, grow, gcol,
                                           make_float4(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1]),
                                                       __uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                           make_float4(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]),
                                                       __uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                        }
                    }
                } else {
                    float *base = S + (static_cast<size_t>(col0 >> 3) * MK_BM + row) * 8;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float x[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(v[8 * q + j]);
                        st_f8_hint(base + q * MK_BM * 8, x, pol);
                    }
                }
                epilogue_pace(p);
            }
        }
        release(acc);
        next_acc();
    }
    bar_sync(1, MK_EPI_THREADS);   // every store of the running sum (or of the output) has been issued
    if (etid == 0 && folded) {
        if (exists) st_release_gpu(p.flags + static_cast<size_t>(lt) * p.P + (r0 + nr - 1), epoch);
        atomicAdd(&c.hdr->units_done, 1u);
        if (exists && last) atomicAdd(&c.hdr->tiles_done, 1u);
    }
    return true;
}

template <int BN>
__device__ void run2_epilogue(const MkParams &p, SmemCtl<Cfg2<BN>::STAGES> &s, uint8_t *stages, const Ctx &c,
                              uint32_t tmem_base, uint32_t epoch, uint32_t crank) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int etid = threadIdx.x - MK_EPI_WARP0 * 32;
    Staging st{stages, Cfg2<BN>::STAGES * Cfg2<BN>::STAGE_BYTES, s.rfull, 0};
    const bool leader = crank == 0;
    const uint32_t tempty0 = mapa_shared(smem_u32(&s.tempty[0]), 0);
    const uint32_t wempty0 = mapa_shared(smem_u32(&s.wempty[0]), 0);
    int acc = 0, wq = 0;
    uint32_t aphase = 0, wphase = 0;
    for (;;) {
        bool ok = true;
        if (lane == 0) ok = wait_bar<true>(smem_u32(&s.wfull[wq]), wphase, c, SITE_WORK_FULL, 0);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!bar_and(1, MK_EPI_THREADS, ok)) break;
        const int2 it = s.items[wq];
        __syncwarp();
        if (lane == 0) {
            if (leader) mbar_arrive(smem_u32(&s.wempty[wq]));
            else mbar_arrive_cluster(wempty0 + 8u * wq);
        }
        if (++wq == WQ) {
            wq = 0;
            wphase ^= 1u;
        }
        if (it.x == ITEM_END) break;
        if (BN == 128 && it.x == ITEM_COMPUTE && p.chain_owner) {
            if (!owner_tile<BN>(p, s, c, tmem_base, it.y, crank, warp, lane, etid, acc, aphase, tempty0)) break;
        } else if (it.x == ITEM_COMPUTE && p.chain_ranks > 1) {
            if (!chain_span<BN>(p, s, c, tmem_base, it.y, crank, warp, lane, etid, acc, aphase, tempty0, epoch)) break;
        } else if (it.x == ITEM_COMPUTE) {
            const int u = it.y;
            int r, sm, tn;
            unit_coords(p, p.pair_tiles_m, u, sm, tn, r);
            const int tm = 2 * sm + static_cast<int>(crank);
            const bool exists = tm < p.tiles_m;
            const int lt = tm * p.tiles_n + tn;
            ok = true;
            if (lane == 0) ok = wait_bar<false>(smem_u32(&s.tfull[acc]), aphase, c, SITE_ACC_FULL, u);
            ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
            if (!bar_and(1, MK_EPI_THREADS, ok)) break;
            tc_fence_after();
            const bool accumulate = p.mode == MK_MODE_ACCUMULATE;
            const bool chained = p.mode == MK_MODE_CHAINED;
            bool folded = true;
            if (exists) {
                if (p.op == MK_IOP_AG)
                    store_output_tile<BN>(p, tmem_base + static_cast<uint32_t>(acc * BN), r, tm, tn, warp, lane);
                else if (accumulate)
                    accumulate_partial<BN>(p, tmem_base + static_cast<uint32_t>(acc * BN), lt, r, warp, lane);
                else if (chained)
                    folded = chain_partial<BN>(p, c, tmem_base + static_cast<uint32_t>(acc * BN), r, tm, tn, warp,
                                               lane, etid, epoch);
                else
                    store_partial<BN>(p, tmem_base + static_cast<uint32_t>(acc * BN), r, lt, warp, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(smem_u32(&s.tempty[acc]));
                else mbar_arrive_remote(tempty0 + 8u * acc);
            }
            if (++acc == ACC) {
                acc = 0;
                aphase ^= 1u;
            }
            if (accumulate) {
                if (exists) finish_accumulate<BN>(p, c, tm, tn, etid);
                if (etid == 0) atomicAdd(&c.hdr->units_done, 1u);
            } else {
                bar_sync(1, MK_EPI_THREADS);   // every store of this partial tile has been issued
                if (etid == 0 && folded) {
                    if (exists && p.op != MK_IOP_AG)
                        st_release_gpu(p.flags + static_cast<size_t>(lt) * p.P + r, epoch);
                    atomicAdd(&c.hdr->units_done, 1u);
                    if (exists && chained && r == p.P - 1) atomicAdd(&c.hdr->tiles_done, 1u);
                }
            }
        } else {
            if (p.op == MK_IOP_AG) {
                int dst, y;
                ag_item(p, it.y, dst, y);
                do_copy_chunk(p, c, 2 * y + static_cast<int>(crank), dst, etid, epoch, st);
            } else {
                int sm, tn;
                raster(it.y / p.red_split, p.pair_tiles_m, p.tiles_n, p.raster_group, sm, tn);
                do_reduce<BN>(p, c, 2 * sm + static_cast<int>(crank), tn, it.y % p.red_split, p.red_split, etid,
                              epoch, st);
            }
        }
        if (etid == 0) *reinterpret_cast<volatile uint32_t *>(&s.epi_done) = s.epi_done + 1;
    }
}

// Run by the even CTA's thread 0 between two cluster barriers at exit: make sure every K-slice
// load either producer issued has landed.  Both producers issue loads in the same stage order,
// so load i uses full[i % STAGES] in phase (i / STAGES) & 1, and only the last STAGES loads can
// be outstanding.  A load armed by one producer only (the other stopped after a pipeline
// timeout) gets the missing arrival here, so its phase completes once its bytes land.
template <int STAGES>
__device__ void pair_drain_loads(SmemCtl<STAGES> &s, const Ctx &c) {
    const uint32_t nl = s.issued, np = s.peer_issued;
    const uint32_t n = nl > np ? nl : np;
    for (uint32_t i = n > STAGES ? n - STAGES : 0; i < n; ++i) {
        const uint32_t bar = smem_u32(&s.full[i % STAGES]);
        if (i >= nl) mbar_arrive(bar);
        if (i >= np) mbar_arrive(bar);
        wait_bar<false>(bar, (i / STAGES) & 1u, c, SITE_DRAIN, i);
    }
}

template <int BN>
__global__ void __launch_bounds__(MK_THREADS, 1) mk_pair_kernel(const __grid_constant__ MkParams p) {
    using T = Cfg2<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                  ~static_cast<uintptr_t>(1023));
    SmemCtl<T::STAGES> &s = *reinterpret_cast<SmemCtl<T::STAGES> *>(stages + T::STAGES * T::STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();

    if (threadIdx.x == 0)
        init_barriers<T::STAGES>(s, p, 2, 2 * (MK_EPI_THREADS / 32), 2 * (1 + MK_EPI_THREADS / 32));
    if (warp == 0 && lane == 0)
        for (int r = 0; r < p.P; ++r) {
            prefetch_tmap(&p.tmA[r]);
            prefetch_tmap(&p.tmB[r]);
        }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&s.tmem_base), T::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;
    const uint32_t epoch = s.epoch;
    const Ctx c{p.hdr, &s.abort, p.timeout_ns, 4 * p.timeout_ns};

    if (warp == 0) {
        if (lane == 0) run2_producer<BN>(p, s, stages, c, crank);
    } else if (warp == 1) {
        if (lane == 0 && crank == 0) run2_mma<BN>(p, s, stages, c, tmem_base);
    } else if (warp < MK_CTRL_WARP) {
        run2_epilogue<BN>(p, s, stages, c, tmem_base, epoch, crank);
    } else if (lane == 0 && blockIdx.x == 0 &&
               (p.mode == MK_MODE_ADAPTIVE || (p.mode == MK_MODE_STATIC && p.trace))) {
        run_controller(p, c, p.num_pair_units,
                       2 * (p.op == MK_IOP_AG ? p.P * p.pair_tiles_m : p.num_pair_tiles * p.red_split), 2,
                       gridDim.x >> 1, 2);
    }
    __syncwarp();
    if (threadIdx.x == 0 && crank == 1) st_cluster_u32(mapa_shared(smem_u32(&s.peer_issued), 0), s.issued);
    tc_fence_before();
    cluster_sync();
    if (threadIdx.x == 0 && crank == 0) pair_drain_loads<T::STAGES>(s, c);
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, T::TMEM_COLS);
    if (threadIdx.x == 0) finish_call(p, epoch);
}

// Second kernel of the unfused baseline: reduce every tile after the GEMM kernel finished
// (stream order replaces the readiness flags).
template <int BN>
__global__ void __launch_bounds__(MK_EPI_THREADS, 1) mk_reduce_kernel(const __grid_constant__ MkParams p) {
    // The same staged reduction as the fused kernel's reduce role, one block per SM with a
    // 192 KiB staging ring, so that the baseline differs from the fused kernel only in when the
    // reduction runs.
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t rfull[3];
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&rfull[i]), 1);
        fence_mbar_init();
        s_abort = 0;
    }
    __syncthreads();
    const Ctx c{p.hdr, &s_abort, p.timeout_ns, 4 * p.timeout_ns};
    Staging st{ring, MK_REDUCE_RING_BYTES, rfull, 0};
    const int items = p.num_tiles * p.red_split;
    for (int i = blockIdx.x; i < items; i += gridDim.x) {
        const int lt = i / p.red_split, sub = i % p.red_split;
        reduce_tile_staged<BN>(p, c, lt / p.tiles_n, lt % p.tiles_n, sub, p.red_split, threadIdx.x, st);
        if (p.discard) discard_tile<BN>(p, lt, sub, p.red_split, threadIdx.x, MK_EPI_THREADS);
    }
}

}  // namespace mk

// ------------------------------------------------------------------ host-side launch helpers
template <int BN, bool PAIR>
static size_t smem_bytes_for() {
    if (PAIR) {
        using T = mk::Cfg2<BN>;
        return static_cast<size_t>(T::STAGES) * T::STAGE_BYTES + sizeof(mk::SmemCtl<T::STAGES>) + 1024;
    }
    using T = mk::Cfg1<BN>;
    return static_cast<size_t>(T::STAGES) * T::STAGE_BYTES + sizeof(mk::SmemCtl<T::STAGES>) + 1024;
}

template <int BN, bool PAIR>
static void *kernel_ptr() {
    return PAIR ? reinterpret_cast<void *>(mk::mk_pair_kernel<BN>)
                : reinterpret_cast<void *>(mk::mk_persistent_kernel<BN>);
}

template <int BN, bool PAIR>
static cudaError_t prepare() {
    return cudaFuncSetAttribute(kernel_ptr<BN, PAIR>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem_bytes_for<BN, PAIR>()));
}

// Per-device results of the one-time launch preparation (the kernel's shared-memory opt-in and its
// occupancy), so that a call pays for the occupancy query only once per device.
constexpr int kMaxDevices = 64;

template <int BN, bool PAIR>
static cudaError_t max_ctas(int *ctas) {
    static std::atomic<int> cached[kMaxDevices];   // co-resident blocks + 1; 0 = not yet known
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *ctas = c - 1;
            return cudaSuccess;
        }
    }
    if ((e = prepare<BN, PAIR>()) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (!PAIR) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mk::mk_persistent_kernel<BN>, MK_THREADS,
                                                          smem_bytes_for<BN, PAIR>());
        *ctas = per_sm * sms;
        if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) cached[dev].store(*ctas + 1);
        return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
    cfg.blockDim = dim3(MK_THREADS);
    cfg.dynamicSmemBytes = smem_bytes_for<BN, PAIR>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, mk::mk_pair_kernel<BN>, &cfg);
    *ctas = 2 * clusters;
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) cached[dev].store(*ctas + 1);
    return e;
}

// Whether this process's runtime accepted a cooperative launch of the clustered kernel
// (-1 unknown, 0 no, 1 yes).  Without it, co-residency rests on the occupancy check the host
// makes before every launch, and the bounded device waits turn a starved grid into an error.
static int g_coop_cluster = -1;

template <int BN, bool PAIR>
static cudaError_t launch_bn(const MkParams &p, int num_ctas, cudaStream_t s) {
    if (PAIR && p.cooperative && g_coop_cluster != 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(num_ctas));
        cfg.blockDim = dim3(MK_THREADS);
        cfg.dynamicSmemBytes = smem_bytes_for<BN, PAIR>();
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        cudaError_t e = cudaLaunchKernelEx(&cfg, mk::mk_pair_kernel<BN>, p);
        if (e == cudaSuccess) {
            g_coop_cluster = 1;
            return e;
        }
        if (g_coop_cluster == 1) return e;
        (void)cudaGetLastError();   // configuration error, not sticky: retry without it
        g_coop_cluster = 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_ctas));
    cfg.blockDim = dim3(MK_THREADS);
    cfg.dynamicSmemBytes = smem_bytes_for<BN, PAIR>();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (!PAIR) {
        if (p.cooperative) {
            attr[n].id = cudaLaunchAttributeCooperative;   // all blocks co-resident, or no launch
            attr[n].val.cooperative = 1;
            ++n;
        }
    } else {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    if (PAIR) return cudaLaunchKernelEx(&cfg, mk::mk_pair_kernel<BN>, p);
    return cudaLaunchKernelEx(&cfg, mk::mk_persistent_kernel<BN>, p);
}

size_t mk_persistent_smem_bytes(int bn, bool pair) {
    if (pair) return bn == 256 ? smem_bytes_for<256, true>() : smem_bytes_for<128, true>();
    return bn == 256 ? smem_bytes_for<256, false>() : smem_bytes_for<128, false>();
}

cudaError_t mk_max_persistent_ctas(int bn, bool pair, int *ctas) {
    if (pair) return bn == 256 ? max_ctas<256, true>(ctas) : max_ctas<128, true>(ctas);
    return bn == 256 ? max_ctas<256, false>(ctas) : max_ctas<128, false>(ctas);
}

cudaError_t mk_launch_persistent(const MkParams &p, int bn, bool pair, int num_ctas, cudaStream_t s) {
    if (pair) return bn == 256 ? launch_bn<256, true>(p, num_ctas, s) : launch_bn<128, true>(p, num_ctas, s);
    return bn == 256 ? launch_bn<256, false>(p, num_ctas, s) : launch_bn<128, false>(p, num_ctas, s);
}

cudaError_t mk_launch_reduce(const MkParams &p, int bn, int num_ctas, cudaStream_t s) {
    const int items = p.num_tiles * p.red_split;
    const int grid = num_ctas < items ? num_ctas : items;
    if (grid <= 0) return cudaSuccess;
    const size_t smem = MK_REDUCE_RING_BYTES + 1024;
    cudaError_t e;
    if (bn == 256) {
        e = cudaFuncSetAttribute(mk::mk_reduce_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        mk::mk_reduce_kernel<256><<<grid, MK_EPI_THREADS, smem, s>>>(p);
    } else {
        e = cudaFuncSetAttribute(mk::mk_reduce_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        mk::mk_reduce_kernel<128><<<grid, MK_EPI_THREADS, smem, s>>>(p);
    }
    return cudaGetLastError();
}
