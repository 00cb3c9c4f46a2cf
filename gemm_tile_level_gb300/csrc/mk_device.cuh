// mk_device.cuh -- device-side error handling and bounded waits shared by the persistent
// kernels (mk_kernels.cu, mk_attention.cu).
#pragma once

#include <stdint.h>

#include "mk.h"
#include "mk_internal.h"
#include "mk_ptx.cuh"

namespace mk {

// Which wait gave up (written to the workspace header with MK_ERR_TIMEOUT).
enum {
    SITE_WORK_EMPTY = 1, SITE_WORK_FULL = 2, SITE_STAGE_EMPTY = 3, SITE_STAGE_FULL = 4,
    SITE_ACC_EMPTY = 5, SITE_ACC_FULL = 6, SITE_FLAG = 7, SITE_DRAIN = 8, SITE_GATE = 9,
    SITE_WATCHDOG = 10, SITE_CLAIMED = 11, SITE_ACC_STATE = 12
};

struct Ctx {
    MkWsHeader *hdr;
    volatile int *s_abort;
    uint64_t timeout_ns;     // cross-block waits
    uint64_t pipe_timeout_ns; // waits inside one block's / pair's pipeline
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

// Bounded pipeline wait on a local mbarrier (cluster-scope acquire when `CLUSTER`): false only
// when 4 x timeout has passed or 2^32 polls were made; that raises MK_ERR_TIMEOUT.
template <bool CLUSTER>
__device__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctx &c, uint32_t site, uint32_t index) {
    auto poll = [&]() { return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1; i != 0u; ++i) {
        if (poll()) return true;
        if ((i & 63u) == 0u && globaltimer() - t0 > c.pipe_timeout_ns) break;
    }
    raise_error(c, MK_ERR_TIMEOUT, site, index);
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

// Named-barrier OR over n threads.
__device__ __forceinline__ bool bar_or(uint32_t id, uint32_t n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
        : "memory");
    return r != 0u;
}

}  // namespace mk
