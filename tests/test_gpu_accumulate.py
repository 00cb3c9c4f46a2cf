"""Accumulate mode (MK_SPLIT_ACCUMULATE): compute blocks add their partial tiles into one fp32
accumulator per output tile with L2 reductions, and the P-th contribution writes the output.

The additions land in no fixed order, so integer inputs (exact in fp32 in any order) are
compared bit for bit with the oracle and random inputs within the tolerances; the workspace is
left zeroed after every successful call and reused as is; a workspace that another mode has
dirtied is refused with MK_ERR_INVALID_ARG until it is zeroed again.
"""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gemm_tile_level_gb300 import api, mk
    import gpu_util as gu

TILES = ("pair", "single")


def acc_opts(tiles="pair", **kw):
    fl = kw.pop("flags", 0) | (mk.MK_FLAG_SINGLE_SM_TILES if tiles == "single" else 0)
    return api.make_opts(mk.MK_SPLIT_ACCUMULATE, flags=fl, **kw)


SHAPES = [
    # P, M, N, K_r
    (1, 1, 8, 8),
    (2, 128, 256, 64),
    (3, 130, 136, 72),
    (5, 300, 520, 24),
    (16, 64, 256, 64),
    (7, 384, 768, 136),
    (8, 1100, 1032, 200),
]


@pytest.mark.parametrize("P,M,N,Kr", SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_integer_bit_exact(P, M, N, Kr, out):
    wl = ig.Workload("acc", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, out, seed=P * 7 + M)
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce(A, B), out == "bf16")
    code = mk.MK_BF16 if out == "bf16" else mk.MK_F32
    for tiles in TILES:
        for fl, band in ((0, 0), (mk.MK_FLAG_TILE_MAJOR, 0), (0, 1)):   # rank-major (default), tile-major, 1-row bands
            C = gu.call_ar(Ad, Bd, code, opts=acc_opts(tiles, flags=fl, raster_group=band))
            gu.assert_bit_exact(gu.host_values(C), ref)


@pytest.mark.parametrize("P,M,N,Kr", SHAPES)
def test_random_within_tolerance(P, M, N, Kr):
    wl = ig.Workload("acc", "allreduce", P, M, N, Kr, ig.normal(1.0), ig.normal(1.0 / (P * Kr)), "bf16", seed=5)
    A, B, Ad, Bd = gu.upload(wl)
    ref = oracle.allreduce(A, B)
    for tiles in TILES:
        for code in (mk.MK_F32, mk.MK_BF16):
            C = gu.call_ar(Ad, Bd, code, opts=acc_opts(tiles))
            gu.check_tolerance(gu.host_values(C), ref, out_bf16=(code == mk.MK_BF16))


def test_reducescatter_integer_bit_exact_and_distinct_outputs():
    P, M, N, Kr = 4, 512, 520, 96
    wl = ig.Workload("acc_rs", "reducescatter", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "bf16", seed=3)
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce(A, B), True)
    for tiles in TILES:
        shards = gu.call_rs(Ad, Bd, mk.MK_BF16, opts=acc_opts(tiles))
        gu.assert_bit_exact(np.concatenate([gu.host_values(s) for s in shards]), ref)
    Cs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    gu.call_ar(Ad, Bd, mk.MK_BF16, C=Cs, opts=acc_opts())
    for c in Cs:
        gu.assert_bit_exact(gu.host_values(c), ref)


def test_consecutive_calls_reuse_the_zeroed_accumulator():
    P, M, N, Kr = 8, 640, 1024, 128
    ws = api.workspace(mk.MK_OP_ALLREDUCE, P, M, N, Kr)
    for seed in (1, 2, 3):
        wl = ig.Workload("acc_reuse", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32", seed=seed)
        A, B, Ad, Bd = gu.upload(wl)
        for tiles in TILES:
            C = gu.call_ar(Ad, Bd, mk.MK_F32, opts=acc_opts(tiles), ws=ws)
            gu.assert_bit_exact(gu.host_values(C), oracle.allreduce(A, B))


def test_workspace_dirtied_by_another_mode_is_refused_until_zeroed():
    P, M, N, Kr = 4, 256, 256, 64
    wl = ig.Workload("acc_dirty", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32", seed=9)
    A, B, Ad, Bd = gu.upload(wl)
    ref = oracle.allreduce(A, B)
    ws = api.workspace(mk.MK_OP_ALLREDUCE, P, M, N, Kr)
    gu.assert_bit_exact(gu.host_values(gu.call_ar(Ad, Bd, mk.MK_F32, ws=ws)), ref)   # adaptive split
    C, st = api.gemm_allreduce(Ad, Bd, mk.MK_F32, ws=ws, opts=acc_opts())
    assert st == mk.MK_OK
    assert mk.mk_status_check(ws) == mk.MK_ERR_INVALID_ARG
    ws.zero_()
    gu.assert_bit_exact(gu.host_values(gu.call_ar(Ad, Bd, mk.MK_F32, ws=ws, opts=acc_opts())), ref)


def test_missing_contribution_is_reported_and_dirties_the_workspace():
    # accumulate mode has no waits: a compute unit that never runs (host-side injection) leaves
    # its tile unwritten, which the last block out reports as an internal error
    P, M, N, Kr = 4, 512, 512, 128
    wl = ig.Workload("acc_skip", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32", seed=4)
    A, B, Ad, Bd = gu.upload(wl)
    ws = api.workspace(mk.MK_OP_ALLREDUCE, P, M, N, Kr)
    C, st = api.gemm_allreduce(Ad, Bd, mk.MK_F32, ws=ws, opts=acc_opts(skip_unit=5))
    assert st == mk.MK_OK
    assert mk.mk_status_check(ws) == mk.MK_ERR_INTERNAL
    C, st = api.gemm_allreduce(Ad, Bd, mk.MK_F32, ws=ws, opts=acc_opts())
    assert mk.mk_status_check(ws) == mk.MK_ERR_INVALID_ARG      # the accumulators are not known to be zero
    ws.zero_()
    gu.assert_bit_exact(gu.host_values(gu.call_ar(Ad, Bd, mk.MK_F32, ws=ws, opts=acc_opts())), oracle.allreduce(A, B))


def test_reducescatter_full_size_sampled():
    wl = ig.WORKLOADS["rs_p8_m16384_n8192_k1024"]
    A, B, Ad, Bd = gu.upload(wl)
    rows, cols = gu.sample_indices(wl.M, wl.N, 4096)
    ref = oracle.allreduce_at(A, B, rows, cols)
    shards = gu.call_rs(Ad, Bd, mk.MK_BF16, opts=acc_opts())
    got = gu.host_values(torch.cat(shards, dim=0))[rows, cols]
    rms = float(np.sqrt(np.mean(oracle.allreduce_rows(A, B, 0, 2) ** 2)))
    gu.check_tolerance(got, ref, out_bf16=True, rms_ref=rms)


def test_allgather_rejects_accumulate():
    Ad = [torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Bd = [torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    _, _, st = api.allgather_gemm(Ad, Bd, mk.MK_F32, opts=acc_opts())
    assert st == mk.MK_ERR_INVALID_ARG
