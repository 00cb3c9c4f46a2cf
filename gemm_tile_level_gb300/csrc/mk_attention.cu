// mk_attention.cu -- Ring Attention (sequence parallelism) for sm_103a: one persistent kernel
// whose blocks either forward KV tiles around the ring (communication role) or run the
// attention of 512 query rows per SM pair against the whole sequence's KV, slice by slice in
// ring order (compute role).
//
// Method (mKernel: Fast Multi-GPU, Multi-Node Fused Kernels; Table 3, row "Ring Attention (SP)";
// abstract, Figure 2): the sequence is cut into P slices, one per rank.  At ring step s rank r
// attends with its own queries to the KV slice of rank (r - s) mod P while that slice moves on to
// rank r + 1; the computations of one step are independent of each other, and KV moves in
// 128-row tiles.  Here the P ranks are P partitions of one GPU's memory.  Communication blocks
// forward each 128-row KV tile from rank r-1's buffer into rank r's ring buffer (bulk copies
// through shared memory) and release a readiness flag per tile; compute blocks acquire the flag
// of each tile before loading it.  Without ring buffers the compute blocks read every slice in
// place.
//
// Compute blocks run as SM pairs (clusters of two, tcgen05 cta_group::2; 352 threads each).  A
// unit is (head h, rank r, 512 query rows) over the P * nt KV tiles of the sequence in ring order
// (step 0 = the rank's own slice): two 256-row query tiles A and B, of which each CTA holds 128
// rows, so that one MMA spans both SMs and each CTA loads only half of every K and V tile.
// Per KV tile j:
//   warp 0    TMA: this CTA's 64 rows of K_j and 64 columns of V_j (16 KiB each, 128-byte swizzle)
//             into a ring of ten slots, in the order K_0, V_0, K_1, V_1, ...
//   warp 1    (even CTA) tcgen05.mma, M = 256 over the pair:
//               O_A += P_A(j) V_j, S_A(j+1) = Q_A K_{j+1}^T, O_B += P_B(j) V_j, S_B(j+1) = Q_B K_{j+1}^T
//             S_A, S_B, O_A, O_B are 128 TMEM columns each (all 512); P_X is read from TMEM
//   warps 2-5 softmax of tile A, warps 6-9 of tile B (one query row per thread = one TMEM lane):
//             running maximum m in the log2 domain, P = 2^(S*scale*log2e - m) as bf16 written back
//             over the first 64 columns of S, row sum l in fp32; when the maximum grows by more
//             than 8 (a factor 256), O and l are rescaled first (otherwise the stale maximum is
//             kept, so P stays below 256)
// and at the end of the unit O / l and lse = (m + log2 l) ln 2 go to memory.
//   warp 10   the communication role inside every compute block: forwards KV tiles around the ring
//             (register copies), claiming them in ring order from a grid-wide counter, so that no
//             SM is taken from the attention.
// Blocks given the communication role outright (a static split) forward tiles from the same
// counter with bulk copies through shared memory; so does every block of the unfused form's
// first kernel.
//
// Every wait is bounded (see mk_device.cuh); a wait that runs out raises MK_ERR_TIMEOUT and
// the grid-wide abort, after which every block drains what it has in flight and exits.
#include "mk.h"
#include "mk_device.cuh"
#include "mk_internal.h"
#include "mk_ptx.cuh"

namespace mk {
namespace attn {

constexpr int BQ = 128;                          // query rows per CTA tile (one TMEM lane each)
constexpr int BKV = 128;                         // KV rows per tile
constexpr int D = MK_ATTN_D;
constexpr uint32_t QBOX = 128 * 64 * 2;          // a 64-column box of 128 rows (16 KiB)
constexpr uint32_t QTILE = 2 * QBOX;             // one CTA's 128 query rows x d
constexpr uint32_t KBOX = 64 * 64 * 2;           // a 64-column box of 64 rows (8 KiB)
constexpr uint32_t SLOT = 16384;                 // one CTA's half of a K tile (64 rows x d) or of a V tile (128 rows x 64)
constexpr int NSLOT = 10;                        // KV ring slots (five KV tiles)
constexpr int COPY_WARPS = 8;                    // warps 2-9 of a communication block
constexpr uint32_t COPY_PIECE = 8192;            // bytes per bulk copy piece
constexpr int COPY_BUFS = 3;                     // staging buffers per copy warp
// SM-pair MMAs (M = 256: each CTA's 128 rows): S = Q K^T with N = 128 KV rows (each CTA supplies 64,
// K-major), O += P V with N = d = 128 (each CTA supplies 64 columns of V, MN-major) and P read from
// tensor memory
constexpr uint32_t IDESC_S = idesc_bf16_f32(2 * BQ, BKV) & ~(1u << 16);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(2 * BQ, D);

// Shared memory (1024-byte aligned): Q_A, Q_B (this CTA's rows), ten 16 KiB KV slots, then control.
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_KV = 2 * QTILE;
constexpr uint32_t DATA_BYTES = OFF_KV + NSLOT * SLOT;
static_assert(COPY_WARPS * COPY_BUFS * COPY_PIECE <= DATA_BYTES, "copy staging fits");

// Barriers.  Those the MMA thread (even CTA) waits on live in the even CTA: q_full and kv_full (two
// producers' expected bytes), p_full and o_free (four softmax warps of each CTA).  Those the MMA
// commits to are multicast to both CTAs: q_empty, kv_empty, s_full, o_done.
struct Ctl {
    uint64_t q_full, q_empty;
    uint64_t kv_full[NSLOT], kv_empty[NSLOT];
    uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
    uint64_t drain;
    uint64_t cbar[COPY_WARPS][COPY_BUFS];
    uint32_t tmem_base;
    uint32_t epoch;
    int abort;
    uint32_t kv_issued, q_issued;              // loads this CTA's producer issued
    uint32_t peer_kv_issued, peer_q_issued;    // even CTA: the odd CTA's counts, stored there at exit
};

static_assert(DATA_BYTES + sizeof(Ctl) + 1024 <= 227 * 1024, "shared memory of one block (227 KiB at most)");

// A unit: head h, rank r, 512 query rows (qp): tile A is rows [0, 256) of it, tile B [256, 512);
// CTA c of the pair holds rows [128 c, 128 c + 128) of each.
struct Unit {
    int h, r, qp;
};

__device__ __forceinline__ Unit unit_of(const MkAttnParams &p, int u) {
    Unit x;
    x.qp = u % p.nq;
    const int hr = u / p.nq;
    x.r = hr % p.P;
    x.h = hr / p.P;
    return x;
}

// Readiness flag of KV tile t of head h that rank r received at ring step s (1 <= s < P).
__device__ __forceinline__ uint32_t *kv_flag(const MkAttnParams &p, int r, int s, int h, int t) {
    return p.flags + ((static_cast<size_t>(r) * (p.P - 1) + (s - 1)) * p.H + h) * p.nt + t;
}

// Wait (bounded) until `f` holds `epoch`, with acquire semantics; false on abort or timeout.
__device__ bool wait_flag(const Ctx &c, const uint32_t *f, uint32_t epoch, uint32_t index) {
    uint64_t t0 = 0;
    for (uint32_t polls = 0; ld_acquire_gpu(f) != epoch; ++polls) {
        if (t0 == 0) t0 = globaltimer();
        if ((polls & 15u) == 15u) {
            if (global_abort(c)) return false;
            if (globaltimer() - t0 > c.timeout_ns || polls > (1u << 30)) {
                raise_error(c, MK_ERR_TIMEOUT, SITE_FLAG, index);
                return false;
            }
        }
        __nanosleep(64);
    }
    return true;
}

// ------------------------------------------------------------------ communication role
// Copy item `item` (ring order: head, then step s = 1..P-1, then receiving rank r, then tile t):
// the K and V rows of KV tile t of head h that rank r receives from rank r-1 at step s.  Its
// source is rank r-1's own K, V at step 1 and, later, what rank r-1 received one step earlier.
struct CopyItem {
    int h, s, r, t, src_rank;
    uint32_t bytes;          // bytes of the K rows (and of the V rows)
    const char *src[2];
    char *dst[2];
};

__device__ __forceinline__ CopyItem copy_item(const MkAttnParams &p, int item) {
    CopyItem x;
    const int per_step = p.P * p.nt;
    const int per_head = (p.P - 1) * per_step;
    x.h = item / per_head;
    const int rem = item - x.h * per_head;
    x.s = rem / per_step + 1;
    const int rem2 = rem - (x.s - 1) * per_step;
    x.r = rem2 / p.nt;
    x.t = rem2 - x.r * p.nt;
    x.src_rank = (x.r + p.P - 1) % p.P;
    const int rows = min(BKV, p.S - x.t * BKV);
    x.bytes = static_cast<uint32_t>(rows) * D * 2;
    const size_t row0 = static_cast<size_t>(x.t) * BKV;
    for (int kv = 0; kv < 2; ++kv) {
        if (x.s == 1)
            x.src[kv] = static_cast<const char *>(kv ? p.v[x.src_rank] : p.k[x.src_rank]) +
                        (static_cast<size_t>(x.h) * p.S + row0) * D * 2;
        else
            x.src[kv] = static_cast<const char *>(p.ring[x.src_rank]) +
                        (((static_cast<size_t>(x.s - 2) * 2 + kv) * p.H + x.h) * p.S + row0) * D * 2;
        x.dst[kv] = static_cast<char *>(p.ring[x.r]) +
                    (((static_cast<size_t>(x.s - 1) * 2 + kv) * p.H + x.h) * p.S + row0) * D * 2;
    }
    return x;
}

// One copy warp forwards KV tile t of head h from rank r-1 to rank r at ring step s: the K and the
// V rows of the tile (contiguous in both buffers) move through three 8 KiB staging buffers with
// bulk copies, then the tile's flag is released.  At step 1 the source is rank r-1's own K_{r-1},
// V_{r-1}; later it is what rank r-1 received one step earlier, so the copy first acquires that
// tile's flag.  Dependencies point to copies with a smaller index only, and every copy warp
// finishes a copy before it starts the next, so the copies always make progress.
__device__ void copy_tile(const MkAttnParams &p, const Ctx &c, int item, uint8_t *stage, uint64_t *bars,
                          uint32_t &seq, uint32_t epoch) {
    const CopyItem x = copy_item(p, item);
    const uint32_t bytes = x.bytes;
    const char *const *src = x.src;
    char *const *dst = x.dst;
    if (x.s >= 2) {
        if (!wait_flag(c, kv_flag(p, x.src_rank, x.s - 1, x.h, x.t), epoch, static_cast<uint32_t>(item))) return;
        fence_proxy_async_global();   // the acquire above before the bulk reads of the source
    }
    const uint32_t npk = (bytes + COPY_PIECE - 1) / COPY_PIECE;   // pieces per K (or V) part
    const uint32_t npieces = 2 * npk;
    auto piece = [&](uint32_t k, const char *&from, char *&to, uint32_t &n) {
        const int kv = k >= npk;
        const uint32_t off = (k - kv * npk) * COPY_PIECE;
        from = src[kv] + off;
        to = dst[kv] + off;
        n = bytes - off < COPY_PIECE ? bytes - off : COPY_PIECE;
    };
    auto load = [&](uint32_t k) {
        const char *from;
        char *to;
        uint32_t n;
        piece(k, from, to, n);
        const uint32_t b = (seq + k) % COPY_BUFS;
        mbar_arrive_expect_tx(smem_u32(&bars[b]), n);
        bulk_load(smem_u32(stage + b * COPY_PIECE), from, n, smem_u32(&bars[b]));
    };
    for (uint32_t k = 0; k < COPY_BUFS - 1 && k < npieces; ++k) load(k);
    for (uint32_t k = 0; k < npieces; ++k) {
        const uint32_t q = seq + k;
        const uint32_t b = q % COPY_BUFS;
        if (!wait_bar<false>(smem_u32(&bars[b]), (q / COPY_BUFS) & 1u, c, SITE_STAGE_FULL, k)) break;
        const char *from;
        char *to;
        uint32_t n;
        piece(k, from, to, n);
        bulk_store(to, smem_u32(stage + b * COPY_PIECE), n);
        bulk_commit();
        if (k + COPY_BUFS - 1 < npieces) {
            bulk_wait_read<COPY_BUFS - 2>();   // the store that last used buffer (k + BUFS - 1) % BUFS has read it
            load(k + COPY_BUFS - 1);
        }
    }
    seq += npieces;
    bulk_wait_all();
    fence_proxy_async_global();        // the bulk writes before the release below
    st_release_gpu(kv_flag(p, x.r, x.s, x.h, x.t), epoch);
}

// Copy items are claimed in ring order from one grid-wide counter by every copy worker (the warps
// of communication blocks, and warp 10 of compute blocks in the fused form).  A copy waits only on
// a copy with a smaller index, which was claimed earlier by a worker that is copying and waits on
// nothing else, so the copies always make progress whatever the compute blocks do.
__device__ __forceinline__ int claim_copy(const MkAttnParams &p) { return static_cast<int>(atomicAdd(&p.hdr->reduce_next, 1u)); }

// A communication block's warp (one thread): bulk copies through its slice of shared memory.
__device__ void run_copies(const MkAttnParams &p, const Ctx &c, Ctl &s, uint8_t *smem, int warp, uint32_t epoch) {
    const int cw = warp - 2;
    uint8_t *stage = smem + static_cast<uint32_t>(cw) * COPY_BUFS * COPY_PIECE;   // a copy block holds no tiles
    uint64_t *bars = s.cbar[cw];
    uint32_t seq = 0;
    for (;;) {
        if (global_abort(c)) break;
        const int item = claim_copy(p);
        if (item >= p.num_copies) break;
        if (item == p.skip_copy) continue;   // fault injection: this tile is never forwarded
        copy_tile(p, c, item, stage, bars, seq, epoch);
    }
    bulk_wait_all();
}

// Warp 10 of a compute block: the same copies with 16-byte register loads and stores, sixteen per
// lane in flight (8 KiB per warp).
__device__ void run_copy_warp(const MkAttnParams &p, const Ctx &c, int lane, uint32_t epoch) {
    constexpr int DEPTH = 16;
    for (;;) {
        int item = 0, stop = 0;
        if (lane == 0) {
            stop = global_abort(c) ? 1 : 0;
            item = stop ? 0 : claim_copy(p);
        }
        stop = __shfl_sync(0xFFFFFFFFu, stop, 0);
        item = __shfl_sync(0xFFFFFFFFu, item, 0);
        if (stop || item >= p.num_copies) break;
        if (item == p.skip_copy) continue;   // fault injection: this tile is never forwarded
        const CopyItem x = copy_item(p, item);
        if (x.s >= 2) {
            int ok = 1;
            if (lane == 0) ok = wait_flag(c, kv_flag(p, x.src_rank, x.s - 1, x.h, x.t), epoch, static_cast<uint32_t>(item));
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;   // lane 0's acquire, then the warp barrier, orders the loads
        }
        const uint32_t n16 = x.bytes / 16;      // 16-byte pieces of the K (or V) rows
        for (int kv = 0; kv < 2; ++kv) {
            const uint4 *from = reinterpret_cast<const uint4 *>(x.src[kv]);
            uint4 *to = reinterpret_cast<uint4 *>(x.dst[kv]);
            for (uint32_t base = 0; base < n16; base += 32 * DEPTH) {
                uint4 v[DEPTH];
#pragma unroll
                for (int k = 0; k < DEPTH; ++k) {
                    const uint32_t i = base + static_cast<uint32_t>(k * 32 + lane);
                    if (i < n16) v[k] = __ldcg(from + i);
                }
#pragma unroll
                for (int k = 0; k < DEPTH; ++k) {
                    const uint32_t i = base + static_cast<uint32_t>(k * 32 + lane);
                    if (i < n16) to[i] = v[k];
                }
            }
        }
        __syncwarp();                           // every lane's stores before lane 0's release
        if (lane == 0) {
            __threadfence();
            st_release_gpu(kv_flag(p, x.r, x.s, x.h, x.t), epoch);
        }
    }
}

// ------------------------------------------------------------------ compute role
// Operand descriptors.  Q (A of S = Q K^T): two 64-column boxes of 128 rows, K-major, 32 bytes per
// 16-column K step.  This CTA's 64 rows of a K tile (B, K-major): two 64-column boxes of 64 rows.
// This CTA's 64 columns of a V tile (B, MN-major: K = KV rows, N = d): one box of 128 rows, 16 rows
// = 2 KiB per K step.
// A descriptor's start address is its low 14-bit field in 16-byte units; every operand here lies
// below 256 KiB of shared memory, so a K step adds its byte offset / 16 to a base descriptor with no
// carry into the other fields.  (Building each descriptor from scratch cost the single issuing
// thread about 85 cycles per MMA, more than an M = 256, N = 128, K = 16 MMA takes.)
__device__ __forceinline__ constexpr uint64_t q_step(int kk) { return ((kk >> 2) * QBOX + (kk & 3) * 32u) >> 4; }
__device__ __forceinline__ constexpr uint64_t k_step(int kk) { return ((kk >> 2) * KBOX + (kk & 3) * 32u) >> 4; }
__device__ __forceinline__ constexpr uint64_t v_step(int kk) { return (kk * 2048u) >> 4; }
__device__ __forceinline__ uint64_t q_desc0(uint32_t tile) { return sw128_desc(tile, 16, 1024); }
__device__ __forceinline__ uint64_t k_desc0(uint32_t slot) { return sw128_desc(slot, 16, 1024); }
__device__ __forceinline__ uint64_t v_desc0(uint32_t slot) { return sw128_desc(slot, SLOT, 1024); }

// Producer (warp 0 of each CTA, one thread): this CTA's rows of Q for each unit, then its halves of
// the KV tiles in the order K_0, V_0, K_1, V_1, ..., counted on the even CTA's barriers.
__device__ void run_producer(const MkAttnParams &p, const Ctx &c, Ctl &s, uint8_t *smem, int pair, int npairs,
                             uint32_t crank, uint32_t epoch) {
    const uint32_t base = smem_u32(smem);
    const int n = p.P * p.nt;
    const uint64_t pol_q = policy_evict_first();
    const uint64_t pol_kv = policy_evict_last();   // every query unit of the head reads them
    const uint32_t q_full0 = mapa_shared(smem_u32(&s.q_full), 0);
    const uint32_t kv_full0 = mapa_shared(smem_u32(&s.kv_full[0]), 0);
    const int half = static_cast<int>(crank);
    uint32_t q = 0, k = 0;
    bool stop = false;
    for (int u = pair; u < p.num_units && !stop; u += npairs, ++k) {
        if (global_abort(c)) break;
        const Unit x = unit_of(p, u);
        if (k > 0 && !wait_bar<false>(smem_u32(&s.q_empty), (k - 1) & 1u, c, SITE_STAGE_EMPTY, u)) break;
        mbar_arrive_expect_tx_cluster(q_full0, 2 * QTILE);
        for (int g = 0; g < 2; ++g)
            for (int box = 0; box < 2; ++box)
                tma_load_3d_pair_hint(base + OFF_Q + g * QTILE + box * QBOX, &p.tmQ[x.r], q_full0, box * 64,
                                      x.qp * 4 * BQ + g * 2 * BQ + half * BQ, x.h, pol_q);
        s.q_issued = k + 1;
        for (int e = 0; e < 2 * n && !stop; ++e) {
            const int j = e >> 1, kind = e & 1;   // kind 0 = this CTA's 64 rows of K_j, 1 = its 64 columns of V_j
            const int st = j / p.nt, t = j - st * p.nt;
            const int o = (x.r - st + p.P) % p.P;
            const bool ring = st > 0 && p.use_ring;
            if (ring && kind == 0 && p.mode == MK_ATTN_FUSED) {
                if (!wait_flag(c, kv_flag(p, x.r, st, x.h, t), epoch, static_cast<uint32_t>(u))) { stop = true; break; }
                fence_proxy_async_global();   // the acquire before the TMA reads of the tile
            }
            const uint32_t slot = q % NSLOT;
            if (q >= NSLOT && !wait_bar<false>(smem_u32(&s.kv_empty[slot]), ((q / NSLOT) - 1) & 1u, c, SITE_STAGE_EMPTY, u)) {
                stop = true;
                break;
            }
            const uint32_t dst = base + OFF_KV + slot * SLOT;
            const uint32_t bar = kv_full0 + 8u * slot;
            mbar_arrive_expect_tx_cluster(bar, SLOT);
            const int z = ring ? ((st - 1) * 2 + kind) * p.H + x.h : x.h;
            if (kind == 0) {
                const CUtensorMap *map = ring ? &p.tmRK[x.r] : &p.tmK[o];
                tma_load_3d_pair_hint(dst, map, bar, 0, t * BKV + half * (BKV / 2), z, pol_kv);
                tma_load_3d_pair_hint(dst + KBOX, map, bar, 64, t * BKV + half * (BKV / 2), z, pol_kv);
            } else {
                const CUtensorMap *map = ring ? &p.tmRV[x.r] : &p.tmV[o];
                tma_load_3d_pair_hint(dst, map, bar, half * 64, t * BKV, z, pol_kv);
            }
            ++q;
            s.kv_issued = q;
        }
    }
}

// MMA issue (warp 1 of the even CTA, one thread).  P_X lives in the first 64 TMEM columns of S_X,
// so S_X(j+1) is issued after O_X += P_X(j) V_j, which MMA issue order keeps behind it.  Per KV
// tile j: O_A += P_A(j) V_j, S_A(j+1), O_B += P_B(j) V_j, S_B(j+1): while one softmax group works,
// the tensor cores run the other group's two MMAs.
__device__ void run_mma(const MkAttnParams &p, const Ctx &c, Ctl &s, uint8_t *smem, uint32_t tmem, int pair,
                        int npairs) {
    const uint32_t base = smem_u32(smem);
    const int n = p.P * p.nt;
    uint32_t q = 0;                  // KV sequence position
    uint32_t np[2] = {0, 0};         // P tiles consumed per group
    uint32_t k = 0;
    bool ok = true;
    auto take = [&](uint32_t &slot) -> bool {   // the next KV half tile of the sequence
        slot = q % NSLOT;
        const bool r = wait_bar<false>(smem_u32(&s.kv_full[slot]), (q / NSLOT) & 1u, c, SITE_STAGE_FULL, q);
        ++q;
        tc_fence_after();
        return r;
    };
    const uint64_t qd[2] = {q_desc0(base + OFF_Q), q_desc0(base + OFF_Q + QTILE)};
    auto issue_s = [&](int g, uint32_t kslot) {
        const uint64_t kd = k_desc0(base + OFF_KV + kslot * SLOT);
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(g) * 128u;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            umma_bf16_pair(d_tmem, qd[g] + q_step(kk), kd + k_step(kk), IDESC_S, static_cast<uint32_t>(kk != 0));
        umma_commit_pair(smem_u32(&s.s_full[g]), 0x3);
    };
    auto issue_pv = [&](int g, uint32_t vslot, bool first) -> bool {
        if (!wait_bar<true>(smem_u32(&s.p_full[g]), np[g] & 1u, c, SITE_ACC_FULL, np[g])) return false;
        ++np[g];
        if (first && k > 0 && !wait_bar<true>(smem_u32(&s.o_free[g]), (k - 1) & 1u, c, SITE_ACC_EMPTY, k)) return false;
        tc_fence_after();
        const uint64_t vd = v_desc0(base + OFF_KV + vslot * SLOT);
        const uint32_t d_tmem = tmem + 256u + static_cast<uint32_t>(g) * 128u;
        const uint32_t a_tmem = tmem + static_cast<uint32_t>(g) * 128u;
        if (first) {
            umma_bf16_pair_ts(d_tmem, a_tmem, vd, IDESC_PV, 0u);
#pragma unroll
            for (int kk = 1; kk < BKV / 16; ++kk)
                umma_bf16_pair_ts(d_tmem, a_tmem + static_cast<uint32_t>(kk) * 8u, vd + v_step(kk), IDESC_PV, 1u);
        } else {
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk)
                umma_bf16_pair_ts(d_tmem, a_tmem + static_cast<uint32_t>(kk) * 8u, vd + v_step(kk), IDESC_PV, 1u);
        }
        return true;
    };
    for (int u = pair; u < p.num_units && ok; u += npairs, ++k) {
        if (!wait_bar<false>(smem_u32(&s.q_full), k & 1u, c, SITE_STAGE_FULL, u)) break;
        tc_fence_after();
        uint32_t ks, vs;
        if (!(ok = take(ks))) break;
        issue_s(0, ks);
        issue_s(1, ks);
        umma_commit_pair(smem_u32(&s.kv_empty[ks]), 0x3);
        if (n == 1) umma_commit_pair(smem_u32(&s.q_empty), 0x3);
        for (int j = 0; j < n && ok; ++j) {
            const bool more = j + 1 < n;
            if (!(ok = take(vs))) break;
            if (!(ok = issue_pv(0, vs, j == 0))) break;
            if (!more) umma_commit_pair(smem_u32(&s.o_done[0]), 0x3);
            if (more) {
                if (!(ok = take(ks))) break;
                issue_s(0, ks);
            }
            if (!(ok = issue_pv(1, vs, j == 0))) break;
            if (!more) umma_commit_pair(smem_u32(&s.o_done[1]), 0x3);
            umma_commit_pair(smem_u32(&s.kv_empty[vs]), 0x3);
            if (more) {
                issue_s(1, ks);
                umma_commit_pair(smem_u32(&s.kv_empty[ks]), 0x3);
                if (j + 2 == n) umma_commit_pair(smem_u32(&s.q_empty), 0x3);   // the unit's last S MMAs are issued
            }
        }
    }
    // every MMA issued must complete before TMEM is released
    umma_commit_pair(smem_u32(&s.drain), 0x1);
    wait_bar<false>(smem_u32(&s.drain), 0, c, SITE_DRAIN, 0);
}

// Two fp32 lanes at once (sm_100 family packed fp32 arithmetic, each lane IEEE-rounded exactly
// as the scalar instruction would be).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// One pass over a row's 128 scores in TMEM (eight 16-column loads): the probabilities
// 2^(s * cl - m) as packed bf16 pairs (columns 2i, 2i+1 in pk[i]), their fp32 sum and the row's
// largest valid score.  With MASK, columns at or past `valid` (the end of the sequence slice)
// count as probability 0.
template <bool MASK>
__device__ __forceinline__ void softmax_pass(uint32_t t_s, int valid, float cl, float m, uint32_t (&pk)[64],
                                             float &rowsum, float &mx) {
    const uint64_t c2 = f2_pack(cl, cl), nm2 = f2_pack(-m, -m);
    uint64_t sum2 = f2_pack(0.0f, 0.0f);
    mx = -INFINITY;
    // the load of chunk cc + 1 is in flight while chunk cc is worked on
    uint32_t buf[2][16];
    tmem_ld16_nowait(t_s, buf[0]);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
        uint32_t (&v)[16] = buf[cc & 1];
        tmem_wait_ld16(v);
        if (cc + 1 < 8) tmem_ld16_nowait(t_s + static_cast<uint32_t>((cc + 1) * 16), buf[(cc + 1) & 1]);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const int col = cc * 16 + i;
            float x0 = __uint_as_float(v[i]), x1 = __uint_as_float(v[i + 1]);
            if (MASK) {
                if (col >= valid) x0 = -INFINITY;
                if (col + 1 >= valid) x1 = -INFINITY;
            }
            mx = max3(mx, x0, x1);
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(x0, x1), c2, nm2), a0, a1);   // s * cl - m, both lanes
            const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);   // 2^-inf = 0 for masked columns
            sum2 = f2_add(sum2, f2_pack(p0, p1));
            pk[col >> 1] = pack_bf16x2(p0, p1);
        }
    }
    float s0, s1;
    f2_unpack(sum2, s0, s1);
    rowsum = s0 + s1;
}

// Softmax group g of a CTA (warps 2-5: g = 0, query tile A; warps 6-9: g = 1, tile B): one query
// row per thread (its TMEM lane).  The running maximum m is only raised when a tile's maximum
// exceeds it by more than 8 (in the log2 domain); otherwise the probabilities are formed against
// the stale maximum (at most 2^8), which needs no first pass for the tile maximum.  A unit's first
// tile takes one (m = -inf), and a row whose tile maximum does exceed m + 8 forms its tile again
// against the new maximum, after O and l are scaled down by 2^(m_old - m_new).  P goes back into the
// first 64 TMEM columns of S as packed bf16 pairs, where the P V MMA reads it.
__device__ void run_softmax(const MkAttnParams &p, const Ctx &c, Ctl &s, uint32_t tmem, int pair, int npairs,
                            uint32_t crank, int g, int warp, int lane) {
    const int quarter = warp & 3;                 // the TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;          // query row in the CTA tile = TMEM lane
    const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lanes + static_cast<uint32_t>(g) * 128u;
    const uint32_t t_o = tmem + lanes + 256u + static_cast<uint32_t>(g) * 128u;
    const uint32_t p_full0 = mapa_shared(smem_u32(&s.p_full[g]), 0);
    const uint32_t o_free0 = mapa_shared(smem_u32(&s.o_free[g]), 0);
    auto arrive_even = [&](uint32_t local_bar, uint32_t even_bar) {   // on the even CTA's barrier
        if (crank == 0) mbar_arrive(local_bar);
        else mbar_arrive_cluster(even_bar);
    };
    const int n = p.P * p.nt;
    const float cl = p.scale_log2;
    uint32_t gt = 0;       // KV tiles processed by this group (all units)
    uint32_t k = 0;
    for (int u = pair; u < p.num_units; u += npairs, ++k) {
        const Unit x = unit_of(p, u);
        float m = -INFINITY, l = 0.0f;
        for (int j = 0, t = 0; j < n; ++j, ++gt, t = (t + 1 == p.nt) ? 0 : t + 1) {   // t = j mod nt
            if (!wait_bar<false>(smem_u32(&s.s_full[g]), gt & 1u, c, SITE_ACC_FULL, gt)) return;
            tc_fence_after();
            const int valid = min(BKV, p.S - t * BKV);
            float alpha = 1.0f;
            if (j == 0) {
                // the unit's first tile: its maximum first
                float mx = -INFINITY;
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t v[32];
                    tmem_ld32(t_s + static_cast<uint32_t>(cc * 32), v);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (cc * 32 + i < valid) mx = fmaxf(mx, __uint_as_float(v[i]));
                }
                m = mx * cl;
                alpha = 0.0f;
            }
            uint32_t pk[64];
            float rowsum;
#pragma unroll 1
            for (int attempt = 0;; ++attempt) {
                float mx;
                if (valid == BKV)
                    softmax_pass<false>(t_s, valid, cl, m, pk, rowsum, mx);
                else
                    softmax_pass<true>(t_s, valid, cl, m, pk, rowsum, mx);
                const float mt = mx * cl;
                const bool grow = attempt == 0 && mt > m + 8.0f;
                if (!__any_sync(0xFFFFFFFFu, grow)) break;
                // rows whose maximum grew past m + 8 form the tile again against it; the other rows
                // of the warp recompute the same values
                if (grow) {
                    alpha = ex2_approx(m - mt);
                    m = mt;
                }
            }
            // every MMA before S(j), the previous P V included, has completed: O may be rescaled
            if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
#pragma unroll 1
                for (int cc = 0; cc < 8; ++cc) {
                    uint32_t ov[16];
                    tmem_ld16(t_o + static_cast<uint32_t>(cc * 16), ov);
#pragma unroll
                    for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    tmem_st16(t_o + static_cast<uint32_t>(cc * 16), ov);
                }
            }
            l = l * alpha + rowsum;
            tmem_st32_nowait(t_s, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st32_nowait(t_s + 32u, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_even(smem_u32(&s.p_full[g]), p_full0);
        }
        // epilogue: O / l and the logsumexp of the unit's query rows
        if (!wait_bar<false>(smem_u32(&s.o_done[g]), k & 1u, c, SITE_ACC_FULL, k)) return;
        tc_fence_after();
        const int qrow = x.qp * 4 * BQ + g * 2 * BQ + static_cast<int>(crank) * BQ + row;
        const bool store = qrow < p.S;
        const size_t obase = (static_cast<size_t>(x.h) * p.S + (store ? qrow : 0)) * D;
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
            uint32_t ov[16];
            tmem_ld16(t_o + static_cast<uint32_t>(cc * 16), ov);
            if (!store) continue;
            float o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __fdiv_rn(__uint_as_float(ov[i]), l);
            if (p.out_bf16) {
                uint16_t *dst = static_cast<uint16_t *>(p.out[x.r]) + obase + cc * 16;
#pragma unroll
                for (int v = 0; v < 2; ++v)
                    st_u4(dst + 8 * v, pack_bf16x2(o[8 * v], o[8 * v + 1]), pack_bf16x2(o[8 * v + 2], o[8 * v + 3]),
                          pack_bf16x2(o[8 * v + 4], o[8 * v + 5]), pack_bf16x2(o[8 * v + 6], o[8 * v + 7]));
            } else {
                float *dst = static_cast<float *>(p.out[x.r]) + obase + cc * 16;
#pragma unroll
                for (int v = 0; v < 4; ++v) st_f4(dst + 4 * v, o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
            }
        }
        if (store && p.lse[x.r]) p.lse[x.r][static_cast<size_t>(x.h) * p.S + qrow] = (m + log2f(l)) * 0.69314718055994531f;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_even(smem_u32(&s.o_free[g]), o_free0);
    }
}

// Last block out records the epoch the call used and resets the per-call state.
__device__ void finish_call(const MkAttnParams &p, uint32_t epoch) {
    MkWsHeader *h = p.hdr;
    __threadfence();
    const uint32_t prev = atomicAdd(&h->done_ctas, 1u);
    if (prev == gridDim.x - 1) {
        __threadfence();
        h->acc_state = MK_ACC_DIRTY;   // the flags are not accumulator tiles of a GEMM call
        h->reduce_next = 0;            // the copy counter
        h->abort = 0;
        h->epoch = epoch;
        h->done_ctas = 0;
        __threadfence();
    }
}

// Run by the even CTA's thread 0 between two cluster barriers at exit: every load either producer
// issued has landed.  Both producers issue the same sequence, so load i of the KV ring uses
// kv_full[i % NSLOT] in phase (i / NSLOT) & 1 and only the last NSLOT can be outstanding; a load
// armed by one producer only (the other stopped after a failed wait) gets the missing arrival here.
__device__ void drain_loads(Ctl &s, const Ctx &c) {
    const uint32_t nl = s.kv_issued, np = s.peer_kv_issued;
    const uint32_t n = nl > np ? nl : np;
    for (uint32_t i = n > NSLOT ? n - NSLOT : 0; i < n; ++i) {
        const uint32_t bar = smem_u32(&s.kv_full[i % NSLOT]);
        if (i >= nl) mbar_arrive(bar);
        if (i >= np) mbar_arrive(bar);
        wait_bar<false>(bar, (i / NSLOT) & 1u, c, SITE_DRAIN, i);
    }
    const uint32_t ql = s.q_issued, qp = s.peer_q_issued;
    const uint32_t qn = ql > qp ? ql : qp;
    if (qn > 0) {
        const uint32_t bar = smem_u32(&s.q_full);
        if (ql < qn) mbar_arrive(bar);
        if (qp < qn) mbar_arrive(bar);
        wait_bar<false>(bar, (qn - 1) & 1u, c, SITE_DRAIN, qn);
    }
}

__global__ void __launch_bounds__(MK_ATTN_THREADS, 1) mk_attn_kernel(const __grid_constant__ MkAttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Ctl &s = *reinterpret_cast<Ctl *>(smem + DATA_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const int npairs_all = static_cast<int>(gridDim.x) >> 1;
    const int ncompute = p.mode == MK_ATTN_COPY_ONLY ? 0
                         : p.mode == MK_ATTN_COMPUTE_ONLY ? npairs_all
                                                          : npairs_all - (p.copy_ctas >> 1);   // compute pairs
    const int pair = static_cast<int>(blockIdx.x) >> 1;
    const bool compute = pair < ncompute;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&s.q_full), 2);
        mbar_init(smem_u32(&s.q_empty), 1);
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(smem_u32(&s.kv_full[i]), 2);
            mbar_init(smem_u32(&s.kv_empty[i]), 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(smem_u32(&s.s_full[g]), 1);
            mbar_init(smem_u32(&s.p_full[g]), 8);
            mbar_init(smem_u32(&s.o_done[g]), 1);
            mbar_init(smem_u32(&s.o_free[g]), 8);
        }
        mbar_init(smem_u32(&s.drain), 1);
        for (int w = 0; w < COPY_WARPS; ++w)
            for (int b = 0; b < COPY_BUFS; ++b) mbar_init(smem_u32(&s.cbar[w][b]), 1);
        fence_mbar_init();
        s.abort = 0;
        s.kv_issued = s.q_issued = s.peer_kv_issued = s.peer_q_issued = 0;
        uint32_t e = ld_relaxed_gpu(&p.hdr->epoch) + 1u;
        if (e == 0u) e = 1u;
        s.epoch = e;
    }
    if (compute && warp == 0 && lane == 0)
        for (int r = 0; r < p.P; ++r) {
            prefetch_tmap(&p.tmQ[r]);
            prefetch_tmap(&p.tmK[r]);
            prefetch_tmap(&p.tmV[r]);
            if (p.use_ring) {
                prefetch_tmap(&p.tmRK[r]);
                prefetch_tmap(&p.tmRV[r]);
            }
        }
    if (compute && warp == 1) {
        tmem_alloc_pair(smem_u32(&s.tmem_base), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t epoch = s.epoch;
    const Ctx c{p.hdr, &s.abort, p.timeout_ns, 4 * p.timeout_ns};

    if (compute) {
        const uint32_t tmem = s.tmem_base;
        if (warp == 0) {
            if (lane == 0) run_producer(p, c, s, smem, pair, ncompute, crank, epoch);
        } else if (warp == 1) {
            if (lane == 0 && crank == 0) run_mma(p, c, s, smem, tmem, pair, ncompute);
        } else if (warp < 10) {
            run_softmax(p, c, s, tmem, pair, ncompute, crank, warp < 6 ? 0 : 1, warp, lane);
        } else if (p.mode == MK_ATTN_FUSED) {
            run_copy_warp(p, c, lane, epoch);
        }
    } else if (warp >= 2 && warp < 2 + COPY_WARPS && lane == 0) {
        run_copies(p, c, s, smem, warp, epoch);
    }
    __syncwarp();
    if (threadIdx.x == 0 && crank == 1) {
        st_cluster_u32(mapa_shared(smem_u32(&s.peer_kv_issued), 0), s.kv_issued);
        st_cluster_u32(mapa_shared(smem_u32(&s.peer_q_issued), 0), s.q_issued);
    }
    tc_fence_before();
    cluster_sync();
    if (compute && threadIdx.x == 0 && crank == 0) drain_loads(s, c);
    cluster_sync();
    tc_fence_after();
    if (compute && warp == 1) tmem_dealloc_pair(s.tmem_base, 512);
    if (threadIdx.x == 0) finish_call(p, epoch);
}

}  // namespace attn
}  // namespace mk

size_t mk_attn_smem_bytes() { return mk::attn::DATA_BYTES + sizeof(mk::attn::Ctl) + 1024; }

cudaError_t mk_attn_max_ctas(int *ctas) {
    static int cached[64] = {};   // co-resident blocks + 1 per device; 0 = not yet known
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) {
        *ctas = cached[dev] - 1;
        return cudaSuccess;
    }
    e = cudaFuncSetAttribute(mk::attn::mk_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(mk_attn_smem_bytes()));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(mk::attn::mk_attn_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
    cfg.blockDim = dim3(MK_ATTN_THREADS);
    cfg.dynamicSmemBytes = mk_attn_smem_bytes();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, mk::attn::mk_attn_kernel, &cfg);
    if (e != cudaSuccess) return e;
    *ctas = 2 * clusters;
    if (dev >= 0 && dev < 64) cached[dev] = *ctas + 1;
    return cudaSuccess;
}

// Whether this process's runtime accepted a cooperative launch of the clustered kernel (-1
// unknown, 0 no, 1 yes); without it co-residency rests on the occupancy check made before every
// launch, and the bounded waits turn a starved grid into an error.
static int g_attn_coop = -1;

cudaError_t mk_launch_attention(const MkAttnParams &p, int num_ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_ctas));
    cfg.blockDim = dim3(MK_ATTN_THREADS);
    cfg.dynamicSmemBytes = mk_attn_smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    if (p.cooperative && g_attn_coop != 0) {
        attr[1].id = cudaLaunchAttributeCooperative;   // every block co-resident, or no launch
        attr[1].val.cooperative = 1;
        cfg.numAttrs = 2;
        cudaError_t e = cudaLaunchKernelEx(&cfg, mk::attn::mk_attn_kernel, p);
        if (e == cudaSuccess) {
            g_attn_coop = 1;
            return e;
        }
        if (g_attn_coop == 1) return e;
        (void)cudaGetLastError();   // configuration error, not sticky: retry without it
        g_attn_coop = 0;
    }
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mk::attn::mk_attn_kernel, p);
}
