// mk_noalloc.cu -- GEMM + AllReduce for callers that cannot allocate device memory.
//
// Some callers of this library have no way to obtain device memory at run time: inference
// runtimes that reserve the whole device up front and hand out nothing more, sandboxed
// plug-ins that are given no allocator, or latency-critical loops where cudaMalloc's implicit
// device-wide synchronisation would stall every other stream.  For them the workspace that
// mk_gemm_allreduce needs (partial tiles, readiness flags, counters) lives in the library
// itself: one file-scope device array per GPU that loads libmk.so, held until the process
// exits.  The caller still owns and passes the operands and the outputs.
#include <cstddef>
#include <cstdio>
#include <mutex>

#include "mk.h"
#include "mk_internal.h"

namespace {

static_assert(MK_ACC_FRESH == 0, "a zeroed header marks the accumulator tiles fresh");

// The library-owned workspace.  In host code `g_noalloc_ws` is only a host-side stand-in for
// the symbol, never a device address: the address is obtained per device below.
static __device__ __align__(256) unsigned char g_noalloc_ws[MK_NOALLOC_MAX_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_ws_ptr[kMaxDevices] = {};   // device address of g_noalloc_ws, per device (null = not set up)

// Once per device, with that device current: resolve the array's device address and zero it,
// so that the workspace header (status, call epoch, counters) starts at zero as mk_gemm_allreduce
// requires.  Synchronous; this is why the first call on a device must precede any stream capture.
mk_status setup_device(int dev, void **out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_ws_ptr[dev]) {
        *out = g_ws_ptr[dev];
        return MK_OK;
    }
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_ws);
    char msg[256];
    if (e != cudaSuccess || !ptr) {
        snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static workspace: %s", cudaGetErrorString(e));
        mk_internal_set_error(msg);
        return MK_ERR_CUDA;
    }
    e = cudaMemset(ptr, 0, MK_NOALLOC_MAX_WS_BYTES);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "zeroing the static workspace: %s", cudaGetErrorString(e));
        mk_internal_set_error(msg);
        return MK_ERR_CUDA;
    }
    g_ws_ptr[dev] = ptr;
    *out = ptr;
    return MK_OK;
}

}  // namespace

extern "C" mk_status mk_gemm_allreduce_noalloc(int P, int64_t M, int64_t N, int64_t K_per_rank,
                                               const void *const *A, const void *const *B, void *const *C,
                                               mk_dtype out_dtype, const mk_opts *opts, void *cuda_stream) {
    const size_t need = mk_workspace_size(MK_OP_ALLREDUCE, P, M, N, K_per_rank);
    if (need > MK_NOALLOC_MAX_WS_BYTES) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "mk_gemm_allreduce_noalloc: this shape needs %zu bytes of workspace; the library's static "
                 "workspace holds %u (use mk_gemm_allreduce with a caller-owned workspace)",
                 need, static_cast<unsigned>(MK_NOALLOC_MAX_WS_BYTES));
        mk_internal_set_error(msg);
        return MK_ERR_WORKSPACE_TOO_SMALL;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        mk_internal_set_error("mk_gemm_allreduce_noalloc: no usable current CUDA device");
        return MK_ERR_CUDA;
    }
    void *ws = nullptr;
    mk_status st = setup_device(dev, &ws);
    if (st != MK_OK) return st;
    // The readiness flags move with the shape, so a previous call's partial tiles may now sit
    // where this call's flags live: clear them (stream-ordered, no allocation).  The header
    // keeps the call epoch and stays as the last call left it.
    const cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    unsigned char *wsb = static_cast<unsigned char *>(ws);
    const size_t flags = need ? mk_internal_flags_bytes(P, M, N, K_per_rank) : 0;
    if (flags && M > 0 && N > 0) {
        e = cudaMemsetAsync(wsb + MK_WS_HEADER_BYTES, 0, flags, stream);
        if (e != cudaSuccess) {
            mk_internal_set_error("mk_gemm_allreduce_noalloc: clearing the flag region failed");
            return MK_ERR_CUDA;
        }
    }
    // An accumulate-mode call adds into fp32 accumulator tiles that must start at zero, and the
    // kernel refuses to run (recording the refusal only in the header, which this entry point
    // never reads) unless the header says they are.  Every other mode leaves partial tiles
    // there, so clear the accumulators and mark them fresh before each accumulate call.
    const bool accumulate = opts && opts->split_mode == MK_SPLIT_ACCUMULATE;
    size_t acc_off = 0, acc_bytes = 0;
    if (accumulate && M > 0 && N > 0 && mk_internal_accumulator_region(P, M, N, K_per_rank, &acc_off, &acc_bytes)) {
        e = cudaMemsetAsync(wsb + acc_off, 0, acc_bytes, stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(wsb + offsetof(MkWsHeader, acc_state), 0, sizeof(uint32_t), stream);   // MK_ACC_FRESH
        if (e != cudaSuccess) {
            mk_internal_set_error("mk_gemm_allreduce_noalloc: clearing the accumulator tiles failed");
            return MK_ERR_CUDA;
        }
    }
    return mk_gemm_allreduce(P, M, N, K_per_rank, A, B, C, out_dtype, ws, MK_NOALLOC_MAX_WS_BYTES, opts,
                             cuda_stream);
}
