// mk_kernels.cu -- the persistent, role-specialised GEMM + reduction kernel for sm_103a
// and the standalone reduction kernel of the unfused baseline.
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
// GB300 mapping of one compute unit (output tile t of rank r, 128 x BN, K_r deep):
//   warp 0  : claims work, TMA-loads 64-wide K slices of A_r and B_r into a 4..6-stage
//             shared-memory ring (128-byte swizzle), completion on mbarriers
//   warp 1  : one thread issues tcgen05.mma (M=128, N=BN, K=16, bf16 -> fp32) into one of two
//             TMEM accumulators and commits to mbarriers
//   warps 2-9: tcgen05.ld the accumulator, store the fp32 partial tile into rank r's
//             workspace partition (coalesced 512-byte warp stores), release flag[t][r]
//   warp 10 : the split controller (block 0, adaptive mode)
// Reduce unit (tile t): warps 2-9 acquire flag[t][0..P-1], stream the P partial tiles with
// 16-byte L2-only loads, sum them in rank order 0..P-1, round and write C (or the shard).
#include "mk_internal.h"
#include "mk_ptx.cuh"
#include "mk.h"

namespace mk {

enum { ITEM_END = 0, ITEM_COMPUTE = 1, ITEM_REDUCE = 2 };

// Which wait gave up (written to the workspace header with MK_ERR_TIMEOUT).
enum {
    SITE_WORK_EMPTY = 1, SITE_WORK_FULL = 2, SITE_STAGE_EMPTY = 3, SITE_STAGE_FULL = 4,
    SITE_ACC_EMPTY = 5, SITE_ACC_FULL = 6, SITE_FLAG = 7, SITE_DRAIN = 8, SITE_GATE = 9,
    SITE_WATCHDOG = 10
};

template <int BN>
struct TileCfg {
    static constexpr int A_BYTES = MK_BM * MK_BK * 2;     // 16 KiB: 128 rows x 128 B
    static constexpr int B_BOX_BYTES = 64 * MK_BK * 2;    // 8 KiB: 64 K rows x 64 N columns
    static constexpr int B_BOXES = BN / 64;
    static constexpr int B_BYTES = B_BOX_BYTES * B_BOXES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (BN == 256) ? 4 : 6;
    static constexpr int ACC = 2;
    static constexpr int TMEM_COLS = ACC * BN;
    static constexpr int WQ = 4;
    static constexpr int TILE_FLOATS = MK_BM * BN;
    static constexpr uint32_t IDESC = idesc_bf16_f32(MK_BM, BN);
};

template <int BN>
struct SmemCtl {
    using T = TileCfg<BN>;
    uint64_t full[T::STAGES];
    uint64_t empty[T::STAGES];
    uint64_t tfull[T::ACC];
    uint64_t tempty[T::ACC];
    uint64_t wfull[T::WQ];
    uint64_t wempty[T::WQ];
    uint64_t drain;
    int2 items[T::WQ];
    uint32_t tmem_base;
    uint32_t epoch;
    int abort;
    int pad;
};

struct Ctx {
    MkWsHeader *hdr;
    volatile int *s_abort;
    uint64_t timeout_ns;
};

__device__ __forceinline__ void raise_error(const Ctx &c, uint32_t code, uint32_t site, uint32_t index) {
    if (atomicCAS(&c.hdr->status, 0u, code) == 0u) {
        c.hdr->err_site = site;
        c.hdr->err_index = index;
    }
    atomicExch(&c.hdr->abort, 1u);
    *c.s_abort = 1;
}

__device__ __forceinline__ bool global_abort(const Ctx &c) {
    if (*c.s_abort) return true;
    if (ld_relaxed_gpu(&c.hdr->abort)) {
        *c.s_abort = 1;
        return true;
    }
    return false;
}

// Bounded mbarrier wait: false if the block is aborting or the limit ran out (which raises
// MK_ERR_TIMEOUT).  At most 2^32 polls and at most timeout_ns.
__device__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctx &c, uint32_t site, uint32_t index) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1; i != 0u; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*c.s_abort) return false;
        if ((i & 63u) == 0u) {
            if (global_abort(c)) return false;
            if (globaltimer() - t0 > c.timeout_ns) break;
        }
    }
    raise_error(c, MK_ERR_TIMEOUT, site, index);
    return false;
}

// Wait used while shutting down: ignores the abort flag (the asynchronous work it waits for
// must finish before the block exits) but keeps the time limit.
__device__ bool wait_bar_final(uint32_t bar, uint32_t parity, const Ctx &c, uint32_t site) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0; i != 0xFFFFFFFFu; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && globaltimer() - t0 > c.timeout_ns) break;
    }
    raise_error(c, MK_ERR_TIMEOUT, site, 0);
    return false;
}

__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
        : "memory");
    return r != 0u;
}

// Grouped raster: groups of `raster_group` tile rows, walked column by column, so that
// concurrently computed tiles share A rows and B columns in L2.
__device__ __forceinline__ void tile_coords(const MkParams &p, int t, int &tm, int &tn) {
    const int G = p.raster_group;
    const int per_group = G * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * G;
    const int gsize = min(G, p.tiles_m - first_m);
    const int local = t - g * per_group;
    tm = first_m + local % gsize;
    tn = local / gsize;
}

// ------------------------------------------------------------------ work claiming
// Role of this block for its next claim: reduce if blockIdx >= S - target (the target is
// published by the controller or fixed by the caller); once the compute queue is empty
// every block reduces.  Block 0 always computes while compute work remains.
//
// Deadlock freedom: a reduction of tile t is queued only after every compute unit of t has
// been claimed (by any block).  Each block works through its queue in claim order, so a
// reduction waits only on units claimed before it, which in turn wait only on items claimed
// earlier still: the wait-for relation follows claim order and has no cycle.
//
// A reduce-role block claims the next tile only when the units finished so far reach it
// (one tile of slack), so that reducers do not park on tiles far ahead of the compute front.
__device__ bool wait_claimed(const MkParams &p, const Ctx &c, uint32_t need) {
    uint64_t t0 = 0;
    for (uint32_t spin = 0; spin != 0xFFFFFFFFu; ++spin) {
        if (ld_relaxed_gpu(&c.hdr->compute_next) >= need) return true;
        if (global_abort(c)) return false;
        if (t0 == 0) t0 = globaltimer();
        else if (globaltimer() - t0 > c.timeout_ns) break;
        __nanosleep(100);
    }
    raise_error(c, MK_ERR_TIMEOUT, SITE_GATE, need);
    return false;
}

__device__ int2 claim_work(const MkParams &p, const Ctx &c, bool &exhausted) {
    MkWsHeader *h = c.hdr;
    const int S = static_cast<int>(gridDim.x);
    const uint32_t num_units = static_cast<uint32_t>(p.num_units);
    const uint32_t P = static_cast<uint32_t>(p.P);
    uint64_t gate_t0 = 0;
    uint32_t gate_seen = 0xFFFFFFFFu;
    for (uint32_t spin = 0; spin != 0xFFFFFFFFu; ++spin) {
        if (global_abort(c)) return make_int2(ITEM_END, 0);
        if (p.mode == MK_MODE_COMPUTE_ONLY) {
            const uint32_t u = atomicAdd(&h->compute_next, 1u);
            if (u >= num_units) return make_int2(ITEM_END, 0);
            if (static_cast<int64_t>(u) == p.skip_unit) continue;
            return make_int2(ITEM_COMPUTE, static_cast<int>(u));
        }
        if (!exhausted) {
            int nr = p.static_nr;
            if (p.mode == MK_MODE_ADAPTIVE) {
                const uint32_t pub = ld_relaxed_gpu(&h->target_nr);
                nr = pub ? static_cast<int>(pub) : p.init_nr;
            }
            if (static_cast<int>(blockIdx.x) < S - nr) {
                const uint32_t u = atomicAdd(&h->compute_next, 1u);
                if (u < num_units) {
                    if (static_cast<int64_t>(u) == p.skip_unit) continue;
                    return make_int2(ITEM_COMPUTE, static_cast<int>(u));
                }
                exhausted = true;
            } else {
                const uint32_t next = ld_relaxed_gpu(&h->reduce_next);
                if (next >= static_cast<uint32_t>(p.num_tiles)) return make_int2(ITEM_END, 0);
                const uint32_t done = ld_relaxed_gpu(&h->units_done);
                const uint32_t issued = ld_relaxed_gpu(&h->compute_next);
                if (issued < num_units &&
                    (static_cast<uint64_t>(next) + 1) * P > static_cast<uint64_t>(done) + P) {
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
        const uint32_t t = atomicAdd(&h->reduce_next, 1u);
        if (t >= static_cast<uint32_t>(p.num_tiles)) return make_int2(ITEM_END, 0);
        const uint64_t need64 = (static_cast<uint64_t>(t) + 1) * P;
        const uint32_t need = need64 < num_units ? static_cast<uint32_t>(need64) : num_units;
        if (!wait_claimed(p, c, need)) return make_int2(ITEM_END, 0);
        return make_int2(ITEM_REDUCE, static_cast<int>(t));
    }
    raise_error(c, MK_ERR_TIMEOUT, SITE_GATE, 0);
    return make_int2(ITEM_END, 0);
}

// ------------------------------------------------------------------ warp 0: scheduler + TMA
template <int BN>
__device__ void run_producer(const MkParams &p, SmemCtl<BN> &s, uint8_t *stages, const Ctx &c) {
    using T = TileCfg<BN>;
    int stage = 0;
    uint32_t phase = 0;
    int wq = 0;
    uint32_t wphase = 0;
    bool exhausted = false;
    uint32_t armed = 0;                 // bit i: stage i has a load issued
    uint32_t armed_phase = 0;           // bit i: phase of that load
    bool stop = false;
    while (!stop) {
        const int2 it = claim_work(p, c, exhausted);
        if (!wait_bar(smem_u32(&s.wempty[wq]), wphase ^ 1u, c, SITE_WORK_EMPTY, 0)) break;
        s.items[wq] = it;
        mbar_arrive(smem_u32(&s.wfull[wq]));
        if (++wq == T::WQ) {
            wq = 0;
            wphase ^= 1u;
        }
        if (it.x == ITEM_END) break;
        if (it.x != ITEM_COMPUTE) continue;
        const int u = it.y;
        const int t = u / p.P;
        const int r = u - t * p.P;
        int tm, tn;
        tile_coords(p, t, tm, tn);
        for (int kb = 0; kb < p.num_kb; ++kb) {
            if (!wait_bar(smem_u32(&s.empty[stage]), phase ^ 1u, c, SITE_STAGE_EMPTY, u)) {
                stop = true;
                break;
            }
            const uint32_t fb = smem_u32(&s.full[stage]);
            uint8_t *sa = stages + stage * T::STAGE_BYTES;
            uint8_t *sb = sa + T::A_BYTES;
            mbar_arrive_expect_tx(fb, T::STAGE_BYTES);
            tma_load_2d(smem_u32(sa), &p.tmA[r], fb, kb * MK_BK, tm * MK_BM);
#pragma unroll
            for (int j = 0; j < T::B_BOXES; ++j)
                tma_load_2d(smem_u32(sb + j * T::B_BOX_BYTES), &p.tmB[r], fb, tn * BN + j * 64,
                            kb * MK_BK);
            armed |= 1u << stage;
            armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == T::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    // Every TMA load issued by this thread must land before the block can exit.
    for (int i = 0; i < T::STAGES; ++i)
        if (armed & (1u << i)) wait_bar_final(smem_u32(&s.full[i]), (armed_phase >> i) & 1u, c, SITE_DRAIN);
}

// ------------------------------------------------------------------ warp 1: tcgen05.mma issue
template <int BN>
__device__ void run_mma(const MkParams &p, SmemCtl<BN> &s, uint8_t *stages, const Ctx &c,
                        uint32_t tmem_base) {
    using T = TileCfg<BN>;
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t aphase = 0;
    int wq = 0;
    uint32_t wphase = 0;
    for (;;) {
        if (!wait_bar(smem_u32(&s.wfull[wq]), wphase, c, SITE_WORK_FULL, 0)) break;
        const int2 it = s.items[wq];
        mbar_arrive(smem_u32(&s.wempty[wq]));
        if (++wq == T::WQ) {
            wq = 0;
            wphase ^= 1u;
        }
        if (it.x == ITEM_END) break;
        if (it.x != ITEM_COMPUTE) continue;
        if (!wait_bar(smem_u32(&s.tempty[acc]), aphase ^ 1u, c, SITE_ACC_EMPTY, it.y)) break;
        tc_fence_after();
        const long long t0 = clock64();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < p.num_kb; ++kb) {
            if (!wait_bar(smem_u32(&s.full[stage]), phase, c, SITE_STAGE_FULL, it.y)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(stages + stage * T::STAGE_BYTES);
            const uint32_t sb = sa + T::A_BYTES;
            // A: K-major, rows 128 B apart, 8-row groups 1024 B apart; K step of 16 = +32 B.
            // B: MN-major, 64-column boxes 8 KiB apart (LBO), 8-row K groups 1024 B apart
            //    (SBO); K step of 16 rows = +2048 B.
            const uint64_t ad = sw128_desc(sa, 16, 1024);
            const uint64_t bd = sw128_desc(sb, T::B_BOX_BYTES, 1024);
#pragma unroll
            for (int kk = 0; kk < MK_BK / 16; ++kk)
                umma_bf16(d_tmem, ad + static_cast<uint64_t>(kk * 2), bd + static_cast<uint64_t>(kk * 128),
                          T::IDESC, static_cast<uint32_t>((kb | kk) != 0));
            umma_commit(smem_u32(&s.empty[stage]));
            if (++stage == T::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        umma_commit(smem_u32(&s.tfull[acc]));
        if (++acc == T::ACC) {
            acc = 0;
            aphase ^= 1u;
        }
        atomicAdd(reinterpret_cast<unsigned long long *>(&c.hdr->compute_busy),
                  static_cast<unsigned long long>(clock64() - t0));
    }
    // Every MMA issued by this thread must complete before TMEM is released.
    umma_commit(smem_u32(&s.drain));
    wait_bar_final(smem_u32(&s.drain), 0, c, SITE_DRAIN);
}

// ------------------------------------------------------------------ reduction of one tile
template <int BN>
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

// Sum the P partial tiles of output tile t in rank order and write the result.  The tile
// layout in a partition is [BN/4 column groups][128 rows][4 floats]; thread `tid` (0..255)
// owns row tid % 128 and one half of the column groups, so each warp load instruction reads
// 512 contiguous bytes.  No waits and no barriers inside.
template <int BN>
__device__ __forceinline__ void reduce_tile_body(const MkParams &p, int t, int tid) {
    using T = TileCfg<BN>;
    int tm, tn;
    tile_coords(p, t, tm, tn);
    const int row = tid & (MK_BM - 1);
    const int grow = tm * MK_BM + row;
    if (grow >= p.M) return;
    const int g_begin = (tid >> 7) * (BN / 8);
    const size_t rank_stride4 = static_cast<size_t>(p.num_tiles) * (T::TILE_FLOATS / 4);
    const float4 *tile4 = reinterpret_cast<const float4 *>(p.partials) +
                          static_cast<size_t>(t) * (T::TILE_FLOATS / 4);
#pragma unroll 1
    for (int g = g_begin; g < g_begin + BN / 8; g += 4) {
        const int gcol = tn * BN + g * 4;
        if (gcol >= p.N) break;
        const float4 *src = tile4 + static_cast<size_t>(g) * MK_BM + row;
        float4 a[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = ld_cg_f4(src + j * MK_BM);
#pragma unroll 1
        for (int r = 1; r < p.P; ++r) {
            const float4 *sr = src + r * rank_stride4;
            float4 x[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = ld_cg_f4(sr + j * MK_BM);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                a[j].x += x[j].x;
                a[j].y += x[j].y;
                a[j].z += x[j].z;
                a[j].w += x[j].w;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (gcol + 4 * j < p.N) store_out4<BN>(p, grow, gcol + 4 * j, a[j]);
    }
}

// Drop the consumed partial tiles of tile t from L2 without write-back (scratch data).
template <int BN>
__device__ __forceinline__ void discard_tile(const MkParams &p, int t, int tid, int nthreads) {
    using T = TileCfg<BN>;
    constexpr int LINES = T::TILE_FLOATS * 4 / 128;
    for (int r = 0; r < p.P; ++r) {
        const char *base = reinterpret_cast<const char *>(
            p.partials + (static_cast<size_t>(r) * p.num_tiles + t) * T::TILE_FLOATS);
        for (int l = tid; l < LINES; l += nthreads) discard_l2_line(base + static_cast<size_t>(l) * 128);
    }
}

// Thread 0 of the reduce group: acquire flag[t][r] == epoch for every rank (bounded).
__device__ bool wait_tile_ready(const MkParams &p, const Ctx &c, int t, uint32_t epoch) {
    const uint32_t *f = p.flags + static_cast<size_t>(t) * p.P;
    uint64_t t0 = 0;
    for (int r = 0; r < p.P; ++r) {
        for (uint32_t polls = 0; ld_acquire_gpu(f + r) != epoch; ++polls) {
            if (*c.s_abort) return false;
            if (t0 == 0) t0 = globaltimer();
            if ((polls & 15u) == 15u) {
                if (global_abort(c)) return false;
                if (globaltimer() - t0 > c.timeout_ns || polls > (1u << 30)) {
                    raise_error(c, MK_ERR_TIMEOUT, SITE_FLAG, static_cast<uint32_t>(t * p.P + r));
                    return false;
                }
            }
            __nanosleep(32);
        }
    }
    return true;
}

// ------------------------------------------------------------------ warps 2-9: epilogue / reduce
template <int BN>
__device__ void run_epilogue(const MkParams &p, SmemCtl<BN> &s, const Ctx &c, uint32_t tmem_base,
                             uint32_t epoch) {
    using T = TileCfg<BN>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int e = warp - MK_EPI_WARP0;
    const int lq = warp & 3;       // the TMEM lane quarter this warp can access
    const int half = e >> 2;       // which half of the tile's columns
    const int etid = threadIdx.x - MK_EPI_WARP0 * 32;
    const int row = lq * 32 + lane;
    int acc = 0;
    uint32_t aphase = 0;
    int wq = 0;
    uint32_t wphase = 0;
    for (;;) {
        bool ok = true;
        if (lane == 0) ok = wait_bar(smem_u32(&s.wfull[wq]), wphase, c, SITE_WORK_FULL, 0);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!bar_and(1, MK_EPI_THREADS, ok)) break;
        const int2 it = s.items[wq];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.wempty[wq]));
        if (++wq == T::WQ) {
            wq = 0;
            wphase ^= 1u;
        }
        if (it.x == ITEM_END) break;
        if (it.x == ITEM_COMPUTE) {
            const int u = it.y;
            const int t = u / p.P;
            const int r = u - t * p.P;
            ok = true;
            if (lane == 0) ok = wait_bar(smem_u32(&s.tfull[acc]), aphase, c, SITE_ACC_FULL, u);
            ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
            if (!bar_and(1, MK_EPI_THREADS, ok)) break;
            tc_fence_after();
            float *tile = p.partials + (static_cast<size_t>(r) * p.num_tiles + t) * T::TILE_FLOATS;
#pragma unroll 1
            for (int cc = 0; cc < BN / 64; ++cc) {
                const int col0 = half * (BN / 2) + cc * 32;
                uint32_t v[32];
                if (p.num_kb > 0) {
                    tmem_ld32(tmem_base + (static_cast<uint32_t>(lq * 32) << 16) +
                                  static_cast<uint32_t>(acc * BN + col0),
                              v);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] = 0u;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float *dst = tile + (static_cast<size_t>((col0 >> 2) + q) * MK_BM + row) * 4;
                    st_f4(dst, __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                          __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.tempty[acc]));
            if (++acc == T::ACC) {
                acc = 0;
                aphase ^= 1u;
            }
            bar_sync(1, MK_EPI_THREADS);   // every store of this partial tile has been issued
            if (etid == 0) {
                st_release_gpu(p.flags + static_cast<size_t>(t) * p.P + r, epoch);
                atomicAdd(&c.hdr->units_done, 1u);
            }
        } else {
            const int t = it.y;
            ok = true;
            if (etid == 0) ok = wait_tile_ready(p, c, t, epoch);
            if (!bar_and(1, MK_EPI_THREADS, ok)) break;
            const long long t0 = clock64();
            reduce_tile_body<BN>(p, t, etid);
            bar_sync(1, MK_EPI_THREADS);   // every read of the partials is done
            if (p.discard) discard_tile<BN>(p, t, etid, MK_EPI_THREADS);
            if (etid == 0) {
                atomicAdd(&c.hdr->tiles_done, 1u);
                atomicAdd(reinterpret_cast<unsigned long long *>(&c.hdr->reduce_busy),
                          static_cast<unsigned long long>(clock64() - t0));
            }
        }
    }
}

// ------------------------------------------------------------------ warp 10: split controller
// Every ctrl_period_ns: with W_c compute units and W_r tiles left, and measured SM-cycle
// costs tau_c per unit and tau_r per tile, publish
//     n_r = clamp(round(S * W_r tau_r / (W_c tau_c + W_r tau_r)), 1, S - 1),
// i.e. give each role SMs in proportion to the work it still has, so both finish together.
// As compute nears completion W_c -> 0 and the target moves toward communication.  This
// formula is a reading of the controller's stated intent; the pages do not give it.
// The loop doubles as a watchdog: no progress for timeout_ns raises MK_ERR_TIMEOUT.
__device__ void run_controller(const MkParams &p, const Ctx &c) {
    MkWsHeader *h = c.hdr;
    const int S = static_cast<int>(gridDim.x);
    int cur = p.init_nr;
    st_relaxed_gpu(&h->target_nr, static_cast<uint32_t>(cur));
    const uint64_t start = globaltimer();
    uint64_t last_change = start;
    uint32_t last_u = 0, last_d = 0;
    mk_trace_record *trace = static_cast<mk_trace_record *>(p.trace);
    uint32_t nrec = 0;
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        const uint32_t u = ld_relaxed_gpu(&h->units_done);
        const uint32_t d = ld_relaxed_gpu(&h->tiles_done);
        const uint64_t now = globaltimer();
        if (trace && nrec < p.trace_cap) {
            mk_trace_record rec;
            rec.t_ns = now - start;
            rec.target = static_cast<uint32_t>(cur);
            rec.units_done = u;
            rec.tiles_done = d;
            rec.num_blocks = static_cast<uint32_t>(S);
            rec.reserved = 0;
            trace[nrec++] = rec;
        }
        if (d >= static_cast<uint32_t>(p.num_tiles) || global_abort(c)) break;
        if (u != last_u || d != last_d) {
            last_u = u;
            last_d = d;
            last_change = now;
        } else if (now - last_change > c.timeout_ns) {
            raise_error(c, MK_ERR_TIMEOUT, SITE_WATCHDOG, d);
            break;
        }
        if (u > 0 && d > 0) {
            const double tau_c = static_cast<double>(ld_relaxed_gpu64(&h->compute_busy)) / u;
            const double tau_r = static_cast<double>(ld_relaxed_gpu64(&h->reduce_busy)) / d;
            const double wc = static_cast<double>(p.num_units - static_cast<int>(min(u, (uint32_t)p.num_units))) * tau_c;
            const double wr = static_cast<double>(p.num_tiles - static_cast<int>(d)) * tau_r;
            int nr = (wc + wr > 0.0) ? static_cast<int>(S * wr / (wc + wr) + 0.5) : cur;
            nr = max(1, min(S - 1, nr));
            if (nr != cur) {
                cur = nr;
                st_relaxed_gpu(&h->target_nr, static_cast<uint32_t>(cur));
            }
        }
        __nanosleep(static_cast<unsigned>(p.ctrl_period_ns));
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
        h->compute_next = 0;
        h->reduce_next = 0;
        h->units_done = 0;
        h->tiles_done = 0;
        h->target_nr = 0;
        h->compute_busy = 0;
        h->reduce_busy = 0;
        h->abort = 0;
        h->epoch = epoch;
        h->done_ctas = 0;
        __threadfence();
    }
}

template <int BN>
__global__ void __launch_bounds__(MK_THREADS, 1) mk_persistent_kernel(const __grid_constant__ MkParams p) {
    using T = TileCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                  ~static_cast<uintptr_t>(1023));
    SmemCtl<BN> &s = *reinterpret_cast<SmemCtl<BN> *>(stages + T::STAGES * T::STAGE_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < T::STAGES; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1);
            mbar_init(smem_u32(&s.empty[i]), 1);
        }
        for (int i = 0; i < T::ACC; ++i) {
            mbar_init(smem_u32(&s.tfull[i]), 1);
            mbar_init(smem_u32(&s.tempty[i]), MK_EPI_THREADS / 32);
        }
        for (int i = 0; i < T::WQ; ++i) {
            mbar_init(smem_u32(&s.wfull[i]), 1);
            mbar_init(smem_u32(&s.wempty[i]), 1 + MK_EPI_THREADS / 32);
        }
        mbar_init(smem_u32(&s.drain), 1);
        fence_mbar_init();
        s.abort = 0;
        uint32_t e = ld_relaxed_gpu(&p.hdr->epoch) + 1u;
        if (e == 0u) e = 1u;
        s.epoch = e;
    }
    if (warp == 0 && lane == 0) {
        for (int r = 0; r < p.P; ++r) {
            prefetch_tmap(&p.tmA[r]);
            prefetch_tmap(&p.tmB[r]);
        }
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
    Ctx c{p.hdr, &s.abort, p.timeout_ns};

    if (warp == 0) {
        if (lane == 0) run_producer<BN>(p, s, stages, c);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) run_mma<BN>(p, s, stages, c, tmem_base);
        __syncwarp();
    } else if (warp < MK_CTRL_WARP) {
        run_epilogue<BN>(p, s, c, tmem_base, epoch);
        __syncwarp();
    } else {
        if (lane == 0 && blockIdx.x == 0 && p.mode == MK_MODE_ADAPTIVE) run_controller(p, c);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, T::TMEM_COLS);
    if (threadIdx.x == 0) finish_call(p, epoch);
}

// Second kernel of the unfused baseline: reduce every tile after the GEMM kernel finished
// (stream order replaces the readiness flags).
template <int BN>
__global__ void __launch_bounds__(MK_EPI_THREADS) mk_reduce_kernel(const __grid_constant__ MkParams p) {
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
        reduce_tile_body<BN>(p, t, threadIdx.x);
        __syncthreads();
        if (p.discard) discard_tile<BN>(p, t, threadIdx.x, MK_EPI_THREADS);
    }
}

}  // namespace mk

// ------------------------------------------------------------------ host-side launch helpers
template <int BN>
static size_t smem_bytes_for() {
    using T = mk::TileCfg<BN>;
    return static_cast<size_t>(T::STAGES) * T::STAGE_BYTES + sizeof(mk::SmemCtl<BN>) + 1024;
}

size_t mk_persistent_smem_bytes(int bn) { return bn == 256 ? smem_bytes_for<256>() : smem_bytes_for<128>(); }

cudaError_t mk_prepare_kernels(int bn) {
    if (bn == 256)
        return cudaFuncSetAttribute(mk::mk_persistent_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem_bytes_for<256>()));
    return cudaFuncSetAttribute(mk::mk_persistent_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem_bytes_for<128>()));
}

cudaError_t mk_max_persistent_ctas(int bn, int *ctas_per_sm) {
    cudaError_t e = mk_prepare_kernels(bn);
    if (e != cudaSuccess) return e;
    if (bn == 256)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, mk::mk_persistent_kernel<256>,
                                                             MK_THREADS, smem_bytes_for<256>());
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, mk::mk_persistent_kernel<128>, MK_THREADS,
                                                         smem_bytes_for<128>());
}

template <int BN>
static cudaError_t launch_persistent_bn(const MkParams &p, int num_ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_ctas));
    cfg.blockDim = dim3(MK_THREADS);
    cfg.dynamicSmemBytes = smem_bytes_for<BN>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // all blocks co-resident, or no launch
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mk::mk_persistent_kernel<BN>, p);
}

cudaError_t mk_launch_persistent(const MkParams &p, int bn, int num_ctas, cudaStream_t s) {
    return bn == 256 ? launch_persistent_bn<256>(p, num_ctas, s) : launch_persistent_bn<128>(p, num_ctas, s);
}

cudaError_t mk_launch_reduce(const MkParams &p, int bn, int num_ctas, cudaStream_t s) {
    const int grid = num_ctas < p.num_tiles ? num_ctas : p.num_tiles;
    if (grid <= 0) return cudaSuccess;
    if (bn == 256)
        mk::mk_reduce_kernel<256><<<grid, MK_EPI_THREADS, 0, s>>>(p);
    else
        mk::mk_reduce_kernel<128><<<grid, MK_EPI_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}
