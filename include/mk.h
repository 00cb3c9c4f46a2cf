/*
 * mk.h -- C ABI of libmk.so: tile-granular fused GEMM + collective kernels of
 * row- and column-parallel tensor parallelism, run on one GB300 (sm_103a)
 * with the P logical ranks held in separate HBM partitions of that GPU.
 *
 * The operations are the three tensor-parallel kernels of
 * "mKernel: Fast Multi-GPU, Multi-Node Fused Kernels", Table 3:
 *   GEMM + AllReduce      (compute -> communication; every rank gets C)
 *   GEMM + ReduceScatter  (compute -> communication; rank s gets row shard s)
 *   AllGather + GEMM      (communication -> compute; row shards of A gathered)
 * and the persistent-kernel design of its Figure 2: thread blocks take a
 * compute role (write finished tiles to GPU memory and set readiness flags) or
 * a communication role (observe the flags and reduce / move the tiles), and an
 * optional on-GPU controller reads progress counters and publishes the target
 * number of communication blocks (abstract; Figure 2, dashed arrow; Figure 7).
 *
 * Conventions shared by every entry point
 *   - All matrices are row-major with no padding (leading dimension = number
 *     of columns).  bf16 operands; fp32 accumulation; bf16 or fp32 output.
 *   - Pointer-array arguments (A, B, C, ...) are HOST arrays of P DEVICE
 *     pointers, one per logical rank.  Every device pointer must be 16-byte
 *     aligned (TMA requirement) and belong to the current CUDA device.
 *   - The caller owns every device buffer (operands, outputs, workspace).  The
 *     library allocates no device memory and keeps no per-call host state; it
 *     caches only the driver's tensor-map encoder entry point.
 *   - Calls are asynchronous and stream-ordered on `cuda_stream` (a
 *     cudaStream_t, NULL = legacy default stream).  Calls that share one
 *     workspace must be ordered on the GPU (same stream or explicit events).
 *   - Synchronous argument errors return a non-zero mk_status and launch
 *     nothing.  Errors found by the kernel (a bounded wait that ran out, an
 *     internal inconsistency) are written to the workspace status word; the
 *     kernel then exits cleanly.  mk_status_check() reports (and clears) it.
 *   - Supported sizes: 1 <= P <= 16; M, N, K >= 0; N and K (per rank) must be
 *     multiples of 8 (16-byte row pitch for TMA).  M == 0 or N == 0 is a
 *     no-op.  K == 0 yields C = 0.  Ragged tails of M and N (not multiples of
 *     the 128 x 256 output tile) and of K (not a multiple of 64) are handled.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MK_OK = 0,
    MK_ERR_INVALID_ARG = 1,        /* null pointer, P out of range, bad option value */
    MK_ERR_UNSUPPORTED_SHAPE = 2,  /* N or K not a multiple of 8, M not divisible by P (RS/AG), too large */
    MK_ERR_ALIGNMENT = 3,          /* a device pointer not 16-byte aligned, workspace not 256-byte aligned */
    MK_ERR_WORKSPACE_TOO_SMALL = 4,/* ws_bytes < mk_workspace_size(...) */
    MK_ERR_CUDA = 5,               /* a CUDA runtime/driver call or the launch failed (see mk_last_error) */
    MK_ERR_TIMEOUT = 6,            /* device side: a bounded wait ran out (wait_timeout_ns) */
    MK_ERR_INTERNAL = 7,           /* device side: inconsistent state detected */
    MK_ERR_NOT_RESIDENT = 8        /* the persistent grid cannot be co-resident on this device */
} mk_status;

typedef enum { MK_BF16 = 0, MK_F32 = 1 } mk_dtype;

typedef enum { MK_OP_ALLREDUCE = 0, MK_OP_REDUCESCATTER = 1, MK_OP_ALLGATHER_GEMM = 2 } mk_op;

typedef enum {
    MK_SPLIT_ADAPTIVE = 0, /* on-GPU controller publishes the reduce-role block count at run time */
    MK_SPLIT_STATIC = 1,   /* comm_sms blocks hold the communication role for the whole call */
    MK_SPLIT_UNFUSED = 2,  /* baseline: one kernel computes every per-rank tile, a second kernel reduces */
    MK_SPLIT_ACCUMULATE = 3, /* no reduce role: compute blocks add their partial tiles into one fp32
                               accumulator tile per output tile with L2 reductions; the last of the
                               P contributions writes the output (AllReduce and ReduceScatter only).
                               The order of the additions is not fixed: exact for integer inputs,
                               within rounding otherwise.  Needs a workspace whose accumulator
                               region is zero: freshly zeroed, or last used by an accumulate call
                               that succeeded; otherwise the call does nothing and
                               mk_status_check reports MK_ERR_INVALID_ARG (zero it again).
                               A tile that did not receive all P contributions is reported
                               as MK_ERR_INTERNAL when the call ends. */
    MK_SPLIT_CHAINED = 4    /* no reduce role: the compute block of (tile, rank r) waits for rank
                               r-1's release, adds its partial tile to the running sum of ranks
                               0..r-1 and stores it (rank P-1 writes the output).  The same fp32
                               additions in the same order as the reduce role, so the same bits
                               (AllReduce and ReduceScatter only).  On SM-pair tiles a compute
                               unit covers chain_ranks consecutive ranks of a tile (all P by
                               default), computed back to back with the running sum kept in
                               tensor memory between them.  For M <= 256 one SM pair computes
                               all P ranks of a 256 x 128 tile and keeps the running sum in
                               tensor memory (the same additions).  MK_FLAG_SINGLE_SM_TILES,
                               or a unit-order flag at M <= 256, selects the one-rank chain on
                               one-SM tiles; debug_skip_unit selects one-rank units at any M. */
} mk_split_mode;

/* Bits of mk_opts.flags */
#define MK_FLAG_KEEP_PARTIALS 1u   /* do not discard consumed partial tiles from L2 (default: discard) */
#define MK_FLAG_SINGLE_SM_TILES 2u /* one SM per 128 x 256 compute tile instead of an SM pair per 256 x 256 */
#define MK_FLAG_NO_L2_HINTS 4u     /* load operands without L2 eviction-priority hints */
#define MK_FLAG_NO_EPILOGUE_PACING 64u /* store each tile's epilogue in one burst (by default the
                                          stores of a tile are spread over part of the next unit's
                                          MMA time, so that they do not hold up its TMA loads) */
#define MK_FLAG_BF16_PARTIALS 128u /* adaptive, static and unfused splits: store each per-rank partial
                                      tile as bf16 (round to nearest even from the fp32 accumulator)
                                      instead of fp32, halving the partial-tile bytes; the reduction
                                      still adds in fp32 in rank order.  The result is then
                                      RNE_out(sum_r RNE_bf16(P_r)): exact on integer inputs whose
                                      per-rank partials are exact in bf16, otherwise within one bf16
                                      rounding per partial.  MK_ERR_INVALID_ARG with the accumulate
                                      and chained splits and with mk_allgather_gemm (no partial
                                      tiles). */
#define MK_FLAG_B_NK 256u         /* GEMM + AllReduce and GEMM + ReduceScatter: each B[r] is given as an
                                     N x K_per_rank row-major matrix (K contiguous: the layout of a linear
                                     layer's weight [out, in]) instead of K_per_rank x N; the operands are
                                     then both K-major for the tensor cores.  The result is the same.
                                     MK_ERR_INVALID_ARG with mk_allgather_gemm. */
#define MK_FLAG_TILE_MAJOR 16u    /* compute the P ranks of each tile back to back */
#define MK_FLAG_RANK_MAJOR 32u    /* compute bands of tile rows rank by rank (see raster_group); without
                                     either flag the order is rank-major for M >= 1024, else tile-major */
#define MK_FLAG_NO_COOPERATIVE 8u  /* launch without the cooperative attribute (some profilers cannot replay
                                      cooperative cluster launches); co-residency then rests on the
                                      occupancy check made before every launch */

/*
 * Options.  Start from mk_opts_default() and change fields; a NULL mk_opts*
 * means the defaults.
 *   split_mode      : mk_split_mode.
 *   comm_sms        : MK_SPLIT_STATIC: number of SMs in the communication role,
 *                     1 <= comm_sms <= grid size - 2 (SM-pair tiles, the
 *                     default, assign roles per pair, so an odd count is
 *                     rounded up to whole pairs; with MK_FLAG_SINGLE_SM_TILES
 *                     roles are per SM and comm_sms <= grid size - 1).
 *                     MK_SPLIT_ADAPTIVE: initial target (0 = one role unit;
 *                     the controller then weighs early against end-of-call
 *                     reduction).  Ignored for MK_SPLIT_UNFUSED, MK_SPLIT_ACCUMULATE
 *                     and MK_SPLIT_CHAINED, which have no reduce role.
 *   wait_timeout_ns : limit of every device-side wait (readiness flags,
 *                     pipeline barriers, the controller's progress watchdog);
 *                     0 = 2 s.  A wait that runs out sets MK_ERR_TIMEOUT.
 *   trace, trace_bytes : optional device buffer receiving controller records
 *                     (mk_trace_record, see below); NULL/0 = off.
 *   num_ctas        : persistent grid size (blocks, one per SM; even with
 *                     SM-pair tiles), 0 = as many as can be co-resident.
 *   flags           : MK_FLAG_* bits.
 *   debug_skip_unit : fault injection for tests: the compute unit (one tile of
 *                     one rank; tiles of 256 rows with SM-pair tiles, of 128
 *                     rows otherwise) with this index in the compute order is
 *                     never produced, so the consumer's bounded wait must run
 *                     out.  -1 = off.
 *   raster_group    : compute tiles are visited in groups ("bands") of this many
 *                     tile rows (256-row rows with SM-pair tiles), column by
 *                     column inside a band, so that the band's A rows stay in
 *                     L2 while B columns stream past them.  In rank-major
 *                     order each band is computed for rank 0, then for rank
 *                     1, ..., so L2 holds one rank's band at a time, and 0
 *                     sizes the band so that one rank's A rows of it take
 *                     about 24 MB.  In tile-major order the P ranks of each
 *                     tile are computed back to back and 0 sizes the band so
 *                     that the A rows of all P ranks take about 32 MB.
 *                     MK_SPLIT_ACCUMULATE computes rank-major unless
 *                     MK_FLAG_TILE_MAJOR is set, and 0 sizes its bands so that
 *                     a band's fp32 accumulator tiles take about 36 MB.
 *   reduce_split    : the reduction of each output tile is cut into this many
 *                     column slices, each claimed as its own item, so that the
 *                     final reductions of a shape with few tiles spread over
 *                     the whole grid; 0 = the smallest power of two (at most
 *                     8) giving every block (SM pair) at least one item, at least
 *                     2 where whole tiles give a block (SM pair) fewer than eight
 *                     items, and at least 2 for the reduce kernel of
 *                     MK_SPLIT_UNFUSED.
 *                     Values above the tile's chunk count (16 for 256-column
 *                     tiles with P <= 8) are clamped to it.  Every element is
 *                     still summed over ranks 0..P-1 in order, so results do
 *                     not depend on it.  Ignored by AllGather + GEMM.
 *   chain_ranks     : MK_SPLIT_CHAINED on SM-pair tiles above M = 256: ranks of a
 *                     tile per compute unit.  The unit computes them back to back
 *                     into the two tensor-memory accumulators in turn, adds the
 *                     running sum read from the workspace to the first, each
 *                     accumulator to the next in place, and stores the sum once;
 *                     0 (or >= P) = all P ranks, so that the running sum never
 *                     leaves tensor memory.  Results do not depend on it.  Ignored
 *                     otherwise; 0 <= chain_ranks <= 16.
 */
typedef struct {
    int32_t split_mode;
    int32_t comm_sms;
    uint64_t wait_timeout_ns;
    void *trace;
    uint64_t trace_bytes;
    int32_t num_ctas;
    uint32_t flags;
    int64_t debug_skip_unit;
    int32_t raster_group;
    int32_t reduce_split;
    int32_t chain_ranks;
} mk_opts;

/* One controller record written to mk_opts.trace (32 bytes). */
typedef struct {
    uint64_t t_ns;          /* time since the controller started */
    uint32_t target;        /* published number of communication-role blocks */
    uint32_t units_done;    /* compute units (tile, rank) finished so far */
    uint32_t tiles_done;    /* output tiles reduced so far */
    uint32_t num_blocks;    /* persistent grid size */
    uint64_t reserved;
} mk_trace_record;

/* Fill *o with the defaults (adaptive split, 2 s waits, no trace, one block per SM). */
void mk_opts_default(mk_opts *o);

/*
 * Bytes of workspace an op needs for this shape (op = mk_op; for
 * MK_OP_ALLGATHER_GEMM, K_per_rank is the full K).  The workspace holds the
 * per-rank fp32 partial tiles (rank r's partition), the readiness flags, the
 * progress counters, the call epoch and the status word.  It must be
 * 256-byte aligned and ZEROED ONCE before its first use; after that it is
 * reused as is (flags are epoch-valued, counters are reset by the kernel).
 * Returns 0 for invalid arguments.
 */
size_t mk_workspace_size(int op, int P, int64_t M, int64_t N, int64_t K_per_rank);

/*
 * GEMM + AllReduce (row-parallel TP): C = sum_{r=0}^{P-1} A_r B_r, delivered
 * to every rank.  (mKernel, Table 3, row "GEMM + AllReduce (TP)": compute ->
 * communication; reduction of the ranks' partial tiles, then broadcast of the
 * result.)
 *   A[r] : M x K_per_rank bf16   (rank r's slice of the activations' K)
 *   B[r] : K_per_rank x N bf16   (rank r's slice of the weight rows; N x K_per_rank with
 *          MK_FLAG_B_NK)
 *   C[r] : M x N, out_dtype      (rank r's copy of the result; entries may
 *                                 alias: each distinct pointer is written once)
 * The sum over ranks is taken in fixed order r = 0, 1, ..., P-1 on fp32
 * partial tiles, so results do not depend on the split mode or timing.
 */
mk_status mk_gemm_allreduce(int P, int64_t M, int64_t N, int64_t K_per_rank,
                            const void *const *A, const void *const *B, void *const *C,
                            mk_dtype out_dtype, void *ws, size_t ws_bytes, const mk_opts *opts,
                            void *cuda_stream);

/*
 * GEMM + ReduceScatter (row-parallel TP): rank s receives rows
 * [s*M/P, (s+1)*M/P) of sum_r A_r B_r.  (mKernel, Table 3, row
 * "GEMM + ReduceScatter (TP)".)  Arguments as for mk_gemm_allreduce except
 *   C_shard[s] : (M/P) x N, out_dtype; M must be divisible by P.
 */
mk_status mk_gemm_reducescatter(int P, int64_t M, int64_t N, int64_t K_per_rank,
                                const void *const *A, const void *const *B, void *const *C_shard,
                                mk_dtype out_dtype, void *ws, size_t ws_bytes, const mk_opts *opts,
                                void *cuda_stream);

/*
 * AllGather + GEMM (column-parallel TP): C_r = [A_0; A_1; ...; A_{P-1}] B_r.
 * (mKernel, Table 3, row "AllGather + GEMM (TP)": communication -> compute,
 * row shards of the activations gathered in 128-row chunks.)
 *   A_shard[s]    : (M/P) x K bf16, rank s's row shard; M divisible by P
 *   B[r]          : K x N bf16, rank r's column shard of the weights
 *   A_gathered[r] : M x K bf16 buffer that receives the gathered activations
 *                   on rank r (all P given), or NULL / all entries NULL: then
 *                   nothing is moved and the compute role reads the shards in
 *                   place (requires M/P to be a multiple of 128)
 *   C[r]          : M x N, out_dtype
 * Communication-role blocks copy 128-row chunks into the gathered buffers,
 * one (chunk, receiving rank) at a time in the order the compute reads them
 * (band by band, rank by rank), and release one readiness flag per chunk and
 * rank; compute-role blocks acquire the flag of the rows they load from their
 * rank's buffer.  The split of SMs between the roles is fixed
 * for the call (comm_sms, or derived from the shape in adaptive mode);
 * MK_SPLIT_UNFUSED gathers in one kernel and multiplies in a second.
 * Workspace: mk_workspace_size(MK_OP_ALLGATHER_GEMM, P, M, N, K).
 */
mk_status mk_allgather_gemm(int P, int64_t M, int64_t N, int64_t K, const void *const *A_shard,
                            const void *const *B, void *const *A_gathered, void *const *C,
                            mk_dtype out_dtype, void *ws, size_t ws_bytes, const mk_opts *opts,
                            void *cuda_stream);

/*
 * Ring Attention (sequence parallelism).  (mKernel, Table 3, row "Ring Attention
 * (SP)": the computations of a ring step are independent of each other; each rank
 * stores its KV slice to the next rank in 128-row tiles; abstract: speedups on Ring
 * Attention.)  The sequence is cut into P contiguous slices of S tokens, one per
 * rank.  At ring step s = 0 .. P-1 rank r attends with its queries to the KV slice
 * of rank (r - s) mod P, which then moves on to rank r + 1, so that after P steps
 * every rank's queries have attended to the whole sequence:
 *   O_r[h][i] = sum over every rank o and key row j of softmax_j(scale * Q_r[h][i] . K_o[h][j]) V_o[h][j]
 * (full, non-causal softmax attention; the pages do not mention a mask).
 *   Q[r], K[r], V[r] : H x S x d bf16, row-major (head-major; each row of d contiguous)
 *   O[r]             : H x S x d, out_dtype
 *   lse[r]           : H x S fp32 natural-log logsumexp of the scaled scores of every
 *                      query row, or lse == NULL / every entry NULL: not written
 *   kv_ring[r]       : (P-1) x 2 x H x S x d bf16 receive buffer of rank r, or
 *                      kv_ring == NULL / every entry NULL.  Given, the call forwards the
 *                      KV around the ring: slot s-1 (s = 1 .. P-1) of rank r receives, from
 *                      rank r-1, the K (index 0) and V (index 1) slice of rank (r - s) mod P,
 *                      one 128-row tile at a time, and the compute reads each step's
 *                      slice from there once its tile's readiness flag is set.  Not given,
 *                      the compute reads every slice in place and nothing is forwarded.
 *   scale            : softmax scale, 0 = 1/sqrt(d)
 *   d                : head dimension; 128 is supported (MK_ERR_UNSUPPORTED_SHAPE otherwise)
 * opts: MK_SPLIT_ADAPTIVE (default) and MK_SPLIT_STATIC run one persistent kernel in
 * which comm_sms blocks (0 = chosen from the shape) forward the KV tiles while the
 * others compute; MK_SPLIT_UNFUSED forwards every step's KV in one kernel and attends
 * in a second.  Other split modes and the GEMM flags are MK_ERR_INVALID_ARG.
 * opts.debug_skip_unit (fault injection for tests): the forwarded KV tile with this index in
 * ring order (head, then step, then receiving rank, then 128-row tile) is never forwarded, so the
 * compute's bounded wait for it runs out (MK_ERR_TIMEOUT from mk_status_check).
 * Arithmetic: scores Q K^T in fp32 from bf16 operands, probabilities as bf16 for P V,
 * fp32 accumulation, an online softmax over the KV tiles in ring order.
 * Workspace: mk_ring_attention_workspace_size(P, H, S, d) bytes, zeroed once (it holds
 * the header and one readiness flag per forwarded tile).
 */
size_t mk_ring_attention_workspace_size(int P, int64_t H, int64_t S, int64_t d);
mk_status mk_ring_attention(int P, int64_t H, int64_t S, int64_t d, const void *const *Q, const void *const *K,
                            const void *const *V, void *const *O, float *const *lse, void *const *kv_ring,
                            mk_dtype out_dtype, float scale, void *ws, size_t ws_bytes, const mk_opts *opts,
                            void *cuda_stream);

/*
 * GEMM + AllReduce without any device allocation by the caller.  The paper has no
 * counterpart to this entry point; it exists for callers that cannot obtain device
 * memory at run time: runtimes that reserve the whole device up front and hand out
 * nothing more, plug-ins that are given no allocator, and latency-critical loops that
 * cannot afford cudaMalloc's implicit device-wide synchronisation.
 *   Arguments and results are those of mk_gemm_allreduce without the workspace: the
 *   library supplies it from one static device array of MK_NOALLOC_MAX_WS_BYTES per
 *   GPU, held from the first call on that GPU until the process exits.  Shapes whose
 *   mk_workspace_size(MK_OP_ALLREDUCE, ...) exceeds that return
 *   MK_ERR_WORKSPACE_TOO_SMALL and launch nothing.
 *   The first call on a device sets the array up (looks up its device address and
 *   zeroes it, synchronously); make that first call before any stream capture.
 *   Every call on a device shares the array and finds the previous call's contents;
 *   each call clears the part that must start at zero.  Calls whose kernels overlap
 *   on the GPU (different streams without ordering, or several host threads) race on
 *   the array and give wrong results: order them.
 *   Every split mode is accepted.  Before an MK_SPLIT_ACCUMULATE call the entry
 *   point also clears the accumulator tiles (stream-ordered memsets), so accumulate
 *   calls work after calls in any other mode.
 *   The return value covers argument, size and launch errors.  What the kernel itself
 *   detects is recorded in the static array and is not reported here: a bounded wait
 *   that ran out (MK_ERR_TIMEOUT: a wait_timeout_ns too short for the shape, or a
 *   withheld unit from debug_skip_unit) and, in accumulate mode, an output tile that
 *   did not receive all P contributions (MK_ERR_INTERNAL).  In either case some output
 *   tiles may be left unwritten.  Callers that need these errors use
 *   mk_gemm_allreduce and mk_status_check with a workspace of their own.
 *   This entry point calls no allocating routine.
 */
#define MK_NOALLOC_MAX_WS_BYTES (64u << 20)
mk_status mk_gemm_allreduce_noalloc(int P, int64_t M, int64_t N, int64_t K_per_rank,
                                    const void *const *A, const void *const *B, void *const *C,
                                    mk_dtype out_dtype, const mk_opts *opts, void *cuda_stream);

/*
 * Synchronize `cuda_stream`, then read and clear the workspace status word.
 * Returns MK_ERR_CUDA if the synchronization itself fails, otherwise the
 * status the kernels recorded since the last check (MK_OK if none).
 */
mk_status mk_status_check(void *ws, void *cuda_stream);

/* Static English description of a status code. */
const char *mk_status_string(mk_status s);

/* Human-readable detail of the last error returned on this host thread ("" if none). */
const char *mk_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MK_H */
