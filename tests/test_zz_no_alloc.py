"""The allocation-free GEMM + AllReduce entry point, mk_gemm_allreduce_noalloc.

It serves callers that cannot get device memory at run time (runtimes that reserve the whole
GPU up front, plug-ins without an allocator, loops that cannot take cudaMalloc's implicit
device-wide synchronisation): the library supplies the workspace from a static device array.
These tests call it through the C ABI and compare its results with those of
mk_gemm_allreduce given a workspace of its own, on consecutive calls that share the static
array (different shapes and output types back to back), and check that a shape too large for
the array is refused.  This file runs last so that a failure here stops a `-x` run only after
every other test has run; it also passes on its own in a fresh process.
"""
import pytest
import torch

import inputgen as ig

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gemm_tile_level_gb300 import mk
    import gpu_util as gu


def _compare_with_workspace_entry_point(wl):
    _, _, Ad, Bd = gu.upload(wl)
    code = mk.MK_BF16 if wl.out_dtype == "bf16" else mk.MK_F32
    want = gu.call_ar(Ad, Bd, code)                      # caller-owned workspace
    got = torch.full_like(want, float("nan"))
    st = mk.mk_gemm_allreduce_noalloc(wl.P, wl.M, wl.N, wl.Kr, Ad, Bd, [got] * wl.P, code)
    mk.check(st)
    torch.cuda.synchronize()
    gu.check_tolerance(gu.host_values(got), gu.host_values(want), out_bf16=(code == mk.MK_BF16))


def test_consecutive_calls_match_the_workspace_entry_point():
    first = ig.Workload("noalloc_a", "allreduce", 4, 512, 1024, 256, ig.normal(1.0), ig.normal(1 / 1024),
                        "bf16", seed=11)
    second = ig.Workload("noalloc_b", "allreduce", 8, 384, 520, 72, ig.UNIFORM_PM1, ig.normal(1 / 576),
                         "f32", seed=12)
    # two calls in a row on different shapes, then the first shape again: each call finds the
    # previous call's contents in the shared static array
    for wl in (first, second, first):
        _compare_with_workspace_entry_point(wl)


def test_shape_beyond_the_static_workspace_is_refused():
    P, M, N, Kr = 8, 2048, 4096, 64
    assert mk.mk_workspace_size(mk.MK_OP_ALLREDUCE, P, M, N, Kr) > mk.MK_NOALLOC_MAX_WS_BYTES
    fake = 0x10000   # never dereferenced: the size check comes before any device work
    st = mk.mk_gemm_allreduce_noalloc(P, M, N, Kr, [fake] * P, [fake] * P, [fake] * P, mk.MK_BF16)
    assert st == mk.MK_ERR_WORKSPACE_TOO_SMALL
    assert "static workspace" in mk.mk_last_error()
