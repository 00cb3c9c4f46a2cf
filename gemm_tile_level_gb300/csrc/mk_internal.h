// mk_internal.h -- layout shared by the host ABI (mk_abi.cu) and the kernels
// (mk_kernels.cu): launch parameters and the workspace header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MK_MAX_P 16

// Output tile of one compute unit is BM x BN; K is consumed in BK slices.
#define MK_BM 128
#define MK_BK 64

// Persistent kernel block: warp 0 schedules and issues TMA loads, warp 1 issues
// tcgen05.mma (and owns the TMEM allocation), warps 2..9 drain accumulators and
// run the reduce role, warp 10 hosts the split controller (block 0 only).
#define MK_THREADS 352
#define MK_EPI_THREADS 256
#define MK_EPI_WARP0 2
#define MK_CTRL_WARP 10

// Workspace layout: [header 256 B][flags][partials]
#define MK_WS_HEADER_BYTES 256
#define MK_WS_ALIGN 256

enum MkMode {
    MK_MODE_ADAPTIVE = 0,   // fused, controller publishes the split
    MK_MODE_STATIC = 1,     // fused, fixed split
    MK_MODE_COMPUTE_ONLY = 2, // unfused baseline: the GEMM kernel
    MK_MODE_COMM_ONLY = 3,    // unfused AllGather baseline: the copy kernel
    MK_MODE_ACCUMULATE = 4,   // compute blocks add their partial tiles into one fp32 accumulator
    MK_MODE_CHAINED = 5       // compute blocks fold their partial tile into a rank-ordered running sum
};

// MkWsHeader::acc_state: whether the accumulator region is known to hold zeros
enum { MK_ACC_FRESH = 0, MK_ACC_CLEAN = 1, MK_ACC_DIRTY = 2 };

enum MkOpInternal { MK_IOP_AR = 0, MK_IOP_RS = 1, MK_IOP_AG = 2 };

// Lives at the start of the workspace; zero-initialised once by the caller.
struct MkWsHeader {
    uint32_t status;        // first device-side error (mk_status), sticky until checked
    uint32_t epoch;         // value the last completed call wrote into the readiness flags
    uint32_t abort;         // set with status; every block stops claiming work
    uint32_t done_ctas;     // blocks finished in the current call
    uint32_t compute_next;  // next compute unit to claim
    uint32_t reduce_next;   // next output tile to claim for reduction
    uint32_t target_nr;     // published number of reduce-role units + 1 (0 = not yet published)
    uint32_t units_done;    // compute units whose partial tile is released
    uint32_t tiles_done;    // output tiles reduced and written
    uint32_t trace_count;   // controller records written
    uint64_t reserved0;     // (unused; keeps the fields below in place)
    uint64_t reduce_busy;   // SM cycles spent reducing ready tiles (sum over blocks)
    uint32_t err_site;      // which wait gave up (diagnostic)
    uint32_t err_index;     // the unit / tile it was waiting for (diagnostic)
    uint32_t acc_state;     // MK_ACC_*: set by every call, read by accumulate-mode calls
    uint32_t pad[(MK_WS_HEADER_BYTES - 68) / 4];
};
static_assert(sizeof(MkWsHeader) == MK_WS_HEADER_BYTES, "workspace header size");

// Launch parameters, passed as one __grid_constant__ kernel argument.
struct MkParams {
    CUtensorMap tmA[MK_MAX_P];   // A_r: dims {K_r, M}, box {64, 128}, 128-byte swizzle
    CUtensorMap tmB[MK_MAX_P];   // B_r: dims {N, K_r}, box {64, 64}; b_nk: dims {K_r, N}, box {64, B rows}; 128-byte swizzle
    void *out[MK_MAX_P];         // AR: distinct result buffers; RS: the P shards
    MkWsHeader *hdr;
    uint32_t *flags;             // [num_tiles][P] readiness flags (epoch-valued)
    float *partials;             // [P][num_tiles][BM*BN] fp32 partial tiles
    void *trace;                 // controller records or null
    int64_t skip_unit;           // fault injection (-1 = off)
    uint64_t timeout_ns;
    uint32_t trace_cap;          // records that fit in trace
    int32_t P, M, N, Kr;
    int32_t tiles_m, tiles_n, num_tiles, num_units, num_kb;
    int32_t pair_tiles_m, num_pair_tiles, num_pair_units;   // SM-pair kernel: 256-row tiles
    int32_t op, out_bf16, num_out, rows_per_shard;
    int32_t mode, static_nr, init_nr, raster_group;
    int32_t discard;
    int32_t l2_hints;            // L2 eviction priorities on partial tiles, running sums and outputs
    int32_t op_hints;            // TMA operand loads: A rows evict_last, B columns evict_first (else normal)
    int32_t cooperative;         // launch attribute (host side only)
    // AllGather + GEMM: A_shard[s] ((M/P) x K) copied in 128-row chunks into every A_gathered[r]
    // (M x K); the compute role waits on the chunk flags (ag_wait) before loading A rows.
    const void *ag_src[MK_MAX_P];
    void *ag_dst[MK_MAX_P];
    int32_t ag_gather, ag_wait;
    int32_t ctrl_period_ns;
    int32_t red_split;           // reduce items per output tile (column slices), >= 1
    int32_t rank_major;          // unit order: 1 = bands of raster_group tile rows, rank by rank
    int32_t ctrl_tail_ns;        // adaptive split: grid time per reduce item at the end of the call
    int32_t epi_pace_ns;         // pause between an epilogue's 32-column store chunks (0 = none)
    int32_t partial_bf16;        // role split / unfused: partial tiles stored as bf16 (RNE), summed in fp32
    int32_t b_nk;                // B_r given as N x K_r (K-major operand; one TMA box of B rows per stage)
    int32_t chain_owner;         // chained mode, short M: one SM pair computes all P ranks of a tile in
                                 // rank order and keeps the running sum in registers (BN = 128 only)
    int32_t band_cols;           // rank-major bands cut into slices of this many tile columns (0 = whole width)
    int32_t chain_ranks;         // chained mode on SM pairs: ranks per compute unit (1, or 2 folded per running-sum pass)
};

// Ring Attention (sequence parallelism): launch parameters of mk_attn_kernel.
enum MkAttnMode {
    MK_ATTN_FUSED = 0,        // copy-role blocks forward KV tiles around the ring, compute blocks attend
    MK_ATTN_COMPUTE_ONLY = 1, // every block attends (the KV it reads is in place, or forwarded earlier)
    MK_ATTN_COPY_ONLY = 2     // every block forwards KV tiles (first kernel of the unfused form)
};

#define MK_ATTN_D 128          // supported head dimension
#define MK_ATTN_THREADS 352    // warp 0 TMA producer, warp 1 MMA, warps 2-9 softmax (two groups of four),
                               // warp 10 forwards KV tiles around the ring

struct MkAttnParams {
    CUtensorMap tmQ[MK_MAX_P];   // Q_r: dims {d, S, H}, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmK[MK_MAX_P];   // K_r: dims {d, S, H}, box {64, 64, 1} (half of a KV tile's rows)
    CUtensorMap tmV[MK_MAX_P];   // V_r: dims {d, S, H}, box {64, 128, 1}
    CUtensorMap tmRK[MK_MAX_P];  // ring buffer of rank r: dims {d, S, (P-1)*2*H}, box {64, 64, 1} (K planes)
    CUtensorMap tmRV[MK_MAX_P];  // the same buffer, box {64, 128, 1} (V planes)
    const void *k[MK_MAX_P];     // K_r, V_r and the ring buffers as plain pointers (bulk copies)
    const void *v[MK_MAX_P];
    void *ring[MK_MAX_P];
    void *out[MK_MAX_P];         // O_r: H x S x d
    float *lse[MK_MAX_P];        // H x S or null
    MkWsHeader *hdr;
    uint32_t *flags;             // [P][P-1][H][nt] readiness of forwarded KV tiles (epoch-valued)
    uint64_t timeout_ns;
    int64_t skip_copy;           // fault injection: the forwarded KV tile never copied (-1 = off)
    float scale_log2;            // softmax scale * log2(e)
    int32_t P, H, S, nt, nq;     // nt: 128-row KV tiles per slice; nq: 512-row query units per slice
    int32_t num_units, num_copies;
    int32_t mode, copy_ctas, use_ring, out_bf16, cooperative;
};

// Implemented in mk_abi.cu: set the host thread's mk_last_error() text; bytes of the readiness
// flag region (which follows the 256-byte header) of the AllReduce workspace for a shape.
void mk_internal_set_error(const char *msg);
size_t mk_internal_flags_bytes(int P, int64_t M, int64_t N, int64_t K_per_rank);
// Offset and bytes of the accumulator tiles an accumulate-mode call (MK_SPLIT_ACCUMULATE) of this
// shape adds into: one fp32 tile per output tile at the start of the partial-tile region.
bool mk_internal_accumulator_region(int P, int64_t M, int64_t N, int64_t K_per_rank, size_t *offset, size_t *bytes);

// Implemented in mk_kernels.cu.  `pair` selects the SM-pair (cta_group::2, 256 x BN) kernel,
// otherwise the one-SM (128 x BN) kernel.
size_t mk_persistent_smem_bytes(int bn, bool pair);
cudaError_t mk_max_persistent_ctas(int bn, bool pair, int *ctas);
cudaError_t mk_launch_persistent(const MkParams &p, int bn, bool pair, int num_ctas, cudaStream_t s);
cudaError_t mk_launch_reduce(const MkParams &p, int bn, int num_ctas, cudaStream_t s);

// Implemented in mk_attention.cu (SM pairs: clusters of two blocks).
size_t mk_attn_smem_bytes();
cudaError_t mk_attn_max_ctas(int *ctas);
cudaError_t mk_launch_attention(const MkAttnParams &p, int num_ctas, cudaStream_t s);
