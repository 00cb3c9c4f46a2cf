"""The allocation-free GEMM + AllReduce entry point, mk_gemm_allreduce_noalloc.

It serves callers that cannot get device memory at run time (runtimes that reserve the whole
GPU up front, plug-ins without an allocator, loops that cannot take cudaMalloc's implicit
device-wide synchronisation): the library supplies the workspace from a static device array
that every call on the GPU shares.  These tests call it through the C ABI:
  * in every split mode, on integer-valued inputs, where the result must equal the oracle bit
    for bit, and on random inputs, where it must equal mk_gemm_allreduce given a workspace of
    its own bit for bit (the same kernel and order), except in accumulate mode, whose order of
    additions is not fixed and which is held to the tolerance instead;
  * on sequences of calls in different modes and shapes back to back, so that each call finds
    what the previous one left in the shared array (partial tiles where accumulate mode expects
    zeroed accumulators, another shape's flags);
  * with a shape too large for the array, which must be refused.
This file runs last so that a failure here stops a `-x` run only after every other test has run;
it also passes on its own in a fresh process.
"""
import pytest
import torch

import inputgen as ig
import oracle

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gemm_tile_level_gb300 import api, mk
    import gpu_util as gu

SPLITS = ("adaptive", "static", "unfused", "chained", "accumulate")


def _opts(split):
    code = {"adaptive": mk.MK_SPLIT_ADAPTIVE, "static": mk.MK_SPLIT_STATIC, "unfused": mk.MK_SPLIT_UNFUSED,
            "chained": mk.MK_SPLIT_CHAINED, "accumulate": mk.MK_SPLIT_ACCUMULATE}[split]
    return api.make_opts(code, comm_sms=8 if split == "static" else 0)


def _noalloc(Ad, Bd, code, split):
    P = len(Ad)
    M, Kr = Ad[0].shape
    N = Bd[0].shape[1]
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16 if code == mk.MK_BF16 else torch.float32,
                     device="cuda")
    mk.check(mk.mk_gemm_allreduce_noalloc(P, M, N, Kr, Ad, Bd, [out] * P, code, opts=_opts(split)))
    torch.cuda.synchronize()
    return out


def _with_own_workspace(Ad, Bd, code, split):
    P = len(Ad)
    M, Kr = Ad[0].shape
    ws = api.workspace(mk.MK_OP_ALLREDUCE, P, M, Bd[0].shape[1], Kr)
    return gu.call_ar(Ad, Bd, code, opts=_opts(split), ws=ws)


def _check_call(wl, split, integer):
    A, B, Ad, Bd = gu.upload(wl, integer=integer)
    code = mk.MK_BF16 if wl.out_dtype == "bf16" else mk.MK_F32
    got = _noalloc(Ad, Bd, code, split)
    if integer:
        # every partial sum is an integer below 2^24: exact in any order, so bit-exact to the oracle
        gu.assert_bit_exact(gu.host_values(got), gu.rounded_reference(oracle.allreduce(A, B), code == mk.MK_BF16))
        return
    want = _with_own_workspace(Ad, Bd, code, split)
    if split == "accumulate":
        gu.check_tolerance(gu.host_values(got), oracle.allreduce(A, B), out_bf16=(code == mk.MK_BF16))
    else:
        assert torch.equal(got, want), f"{split}: differs from mk_gemm_allreduce with its own workspace"


def _workloads():
    first = ig.Workload("noalloc_a", "allreduce", 4, 512, 1024, 256, ig.normal(1.0), ig.normal(1 / 1024),
                        "bf16", seed=11)
    second = ig.Workload("noalloc_b", "allreduce", 8, 384, 520, 72, ig.UNIFORM_PM1, ig.normal(1 / 576),
                         "f32", seed=12)
    return first, second


@pytest.mark.parametrize("split", SPLITS)
def test_each_split_mode_twice_in_a_row(split):
    first, second = _workloads()
    for wl in (first, second):
        _check_call(wl, split, integer=True)
        _check_call(wl, split, integer=False)


@pytest.mark.parametrize("sequence", [
    ("chained", "accumulate", "adaptive"),
    ("adaptive", "accumulate", "accumulate", "unfused"),
    ("unfused", "static", "accumulate", "chained", "accumulate"),
])
def test_mode_changes_on_the_shared_array(sequence):
    first, second = _workloads()
    for i, split in enumerate(sequence):
        wl = (first, second)[i % 2]
        _check_call(wl, split, integer=(i % 2 == 0))


def test_consecutive_calls_match_the_workspace_entry_point():
    first, second = _workloads()
    # two calls in a row on different shapes, then the first shape again: each call finds the
    # previous call's contents in the shared static array
    for wl in (first, second, first):
        _check_call(wl, "adaptive", integer=False)


def test_shape_beyond_the_static_workspace_is_refused():
    P, M, N, Kr = 8, 2048, 4096, 64
    assert mk.mk_workspace_size(mk.MK_OP_ALLREDUCE, P, M, N, Kr) > mk.MK_NOALLOC_MAX_WS_BYTES
    fake = 0x10000   # never dereferenced: the size check comes before any device work
    st = mk.mk_gemm_allreduce_noalloc(P, M, N, Kr, [fake] * P, [fake] * P, [fake] * P, mk.MK_BF16)
    assert st == mk.MK_ERR_WORKSPACE_TOO_SMALL
    assert "static workspace" in mk.mk_last_error()
