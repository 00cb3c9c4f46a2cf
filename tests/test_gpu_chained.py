"""Chained mode (MK_SPLIT_CHAINED): the compute block of (tile, rank r) folds its partial tile
into the running sum of ranks 0..r-1 after rank r-1's release, and rank P-1 writes the output.
On a short M (M <= 256, the default tile kind and order) one SM pair instead owns each tile,
computes its P ranks in turn and keeps the running sum in TMEM; a tile-kind or unit-order flag
selects the rank-ordered chain there too, so both paths are run below.  On SM pairs above one
band a compute unit covers chain_ranks consecutive ranks of a tile (all P by default) whose sum
crosses the workspace once per unit; 1, 2 and 3 ranks per unit with odd P, P = 1 and P = 2 run
its one-rank, first-unit and later-unit cases.

These are the reduce role's fp32 additions in the reduce role's order, so on random inputs the
result must equal the adaptive, static and unfused results bit for bit, besides matching the
oracle (bit-exact on integer inputs).  A withheld compute unit makes its successor's bounded
wait run out.
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


def ch_opts(tiles="pair", **kw):
    fl = kw.pop("flags", 0) | (mk.MK_FLAG_SINGLE_SM_TILES if tiles == "single" else 0)
    return api.make_opts(mk.MK_SPLIT_CHAINED, flags=fl, **kw)


SHAPES = [
    (1, 1, 8, 8),
    (2, 128, 256, 64),
    (3, 130, 136, 72),
    (5, 300, 520, 24),
    (16, 64, 256, 64),
    (7, 384, 768, 136),
    (8, 1100, 1032, 200),
    (5, 1100, 520, 72),    # SM pairs, odd P: the last unit folds one rank
    (1, 640, 264, 64),     # SM pairs, one rank: straight to the output
    (2, 768, 136, 40),     # SM pairs, P = 2: one two-rank unit per tile, ragged N
    (16, 640, 392, 48),    # SM pairs, the most ranks: sixteen folds per unit, ragged M and N
]


@pytest.mark.parametrize("P,M,N,Kr", SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_integer_bit_exact(P, M, N, Kr, out):
    wl = ig.Workload("ch", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, out, seed=P * 5 + M)
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce(A, B), out == "bf16")
    code = mk.MK_BF16 if out == "bf16" else mk.MK_F32
    for tiles in TILES:
        # (0, 0): tile owners when M <= 256 with pair tiles; the order flags force the chain
        for fl, band in ((0, 0), (mk.MK_FLAG_TILE_MAJOR, 0), (mk.MK_FLAG_RANK_MAJOR, 0), (0, 1)):
            C = gu.call_ar(Ad, Bd, code, opts=ch_opts(tiles, flags=fl, raster_group=band))
            gu.assert_bit_exact(gu.host_values(C), ref)
    # SM pairs above one band: 1, 2 and 3 ranks per unit besides the default (all P): the running
    # sum crosses the workspace between units, a unit may hold a single rank
    for cr in (1, 2, 3):
        for fl in (0, mk.MK_FLAG_TILE_MAJOR):
            C = gu.call_ar(Ad, Bd, code, opts=ch_opts(flags=fl, chain_ranks=cr))
            gu.assert_bit_exact(gu.host_values(C), ref)


@pytest.mark.parametrize("P,M,N,Kr", SHAPES)
def test_random_same_bits_as_the_reduce_role(P, M, N, Kr):
    wl = ig.Workload("ch", "allreduce", P, M, N, Kr, ig.normal(1.0), ig.normal(1.0 / (P * Kr)), "f32", seed=6)
    A, B, Ad, Bd = gu.upload(wl)
    ref = oracle.allreduce(A, B)
    for tiles in TILES:
        fl = mk.MK_FLAG_SINGLE_SM_TILES if tiles == "single" else 0
        want = gu.call_ar(Ad, Bd, mk.MK_F32, opts=api.make_opts(mk.MK_SPLIT_UNFUSED, flags=fl))
        for order in (0, mk.MK_FLAG_RANK_MAJOR):
            got = gu.call_ar(Ad, Bd, mk.MK_F32, opts=ch_opts(tiles, flags=order))
            gu.check_tolerance(gu.host_values(got), ref, out_bf16=False)
            assert torch.equal(got, want)
    for cr in (1, 2, 3):
        assert torch.equal(gu.call_ar(Ad, Bd, mk.MK_F32, opts=ch_opts(chain_ranks=cr)), want)


@pytest.mark.parametrize("P,M,N", [(3, 200, 136), (8, 256, 8192), (2, 1024, 512)])
def test_zero_k_gives_zeros(P, M, N):
    Ad = [torch.empty((M, 0), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    Bd = [torch.empty((0, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    for tiles in TILES:
        for order in (0, mk.MK_FLAG_RANK_MAJOR):
            C = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
            gu.call_ar(Ad, Bd, mk.MK_F32, C=C, opts=ch_opts(tiles, flags=order))
            assert not C.any()


@pytest.mark.parametrize("M", [256, 512])
def test_short_m_sweep_shape_both_paths_same_bits(M):
    """The sweep's short shapes (P=8, N=8192, K_r=1024): tile owners (M = 256), SM-pair units of
    several ranks (M = 512) and the one-rank chain on one-SM tiles against the unfused baseline,
    bit for bit, and against the oracle on sampled elements."""
    wl = ig.sweep_workload(M)
    A, B, Ad, Bd = gu.upload(wl)
    want = gu.call_ar(Ad, Bd, mk.MK_BF16, opts=api.make_opts(mk.MK_SPLIT_UNFUSED))
    for fl in (0, mk.MK_FLAG_RANK_MAJOR, mk.MK_FLAG_SINGLE_SM_TILES):
        assert torch.equal(gu.call_ar(Ad, Bd, mk.MK_BF16, opts=ch_opts(flags=fl)), want)
    if M > 256:   # SM-pair units of all 8 ranks by default; of 3 ranks (a short last group) and 2
        for cr in (2, 3):
            assert torch.equal(gu.call_ar(Ad, Bd, mk.MK_BF16, opts=ch_opts(chain_ranks=cr)), want)
    rows, cols = gu.sample_indices(wl.M, wl.N, 1024)
    rms = float(np.sqrt(np.mean(oracle.allreduce_rows(A, B, 0, 2) ** 2)))
    gu.check_tolerance(gu.host_values(want)[rows, cols], oracle.allreduce_at(A, B, rows, cols), out_bf16=True,
                       rms_ref=rms)


@pytest.mark.parametrize("M", [1024, 512, 256])   # SM-pair units of several ranks (1024, 512); tile owners (256)
def test_reducescatter_and_distinct_outputs(M):
    P, N, Kr = 4, 520, 96
    wl = ig.Workload("ch_rs", "reducescatter", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "bf16", seed=3)
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce(A, B), True)
    for tiles in TILES:
        for order in (0, mk.MK_FLAG_RANK_MAJOR):
            shards = gu.call_rs(Ad, Bd, mk.MK_BF16, opts=ch_opts(tiles, flags=order))
            gu.assert_bit_exact(np.concatenate([gu.host_values(s) for s in shards]), ref)
    for cr in (1, 3):
        shards = gu.call_rs(Ad, Bd, mk.MK_BF16, opts=ch_opts(chain_ranks=cr))
        gu.assert_bit_exact(np.concatenate([gu.host_values(s) for s in shards]), ref)
    for order in (0, mk.MK_FLAG_RANK_MAJOR):
        Cs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        gu.call_ar(Ad, Bd, mk.MK_BF16, C=Cs, opts=ch_opts(flags=order))
        for c in Cs:
            gu.assert_bit_exact(gu.host_values(c), ref)


def test_full_size_same_bits_as_the_reduce_role():
    wl = ig.WORKLOADS["ar_mlp_down_p8_m8192_n8192_k3584"]
    A, B, Ad, Bd = gu.upload(wl)
    ws = api.workspace(mk.MK_OP_ALLREDUCE, wl.P, wl.M, wl.N, wl.Kr)
    want = gu.call_ar(Ad, Bd, mk.MK_BF16, ws=ws)
    got = gu.call_ar(Ad, Bd, mk.MK_BF16, ws=ws, opts=ch_opts())
    assert torch.equal(got, want)
    rows, cols = gu.sample_indices(wl.M, wl.N, 2048)
    rms = float(np.sqrt(np.mean(oracle.allreduce_rows(A, B, 0, 2) ** 2)))
    gu.check_tolerance(gu.host_values(got)[rows, cols], oracle.allreduce_at(A, B, rows, cols), out_bf16=True,
                       rms_ref=rms)


@pytest.mark.parametrize("tiles", TILES)
def test_missing_unit_times_out_then_recovers(tiles):
    wl = ig.Workload("ch_fault", "allreduce", 4, 512, 512, 128, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32")
    A, B, Ad, Bd = gu.upload(wl)
    ws = api.workspace(mk.MK_OP_ALLREDUCE, 4, 512, 512, 128)
    C, st = api.gemm_allreduce(Ad, Bd, mk.MK_F32, ws=ws, opts=ch_opts(tiles, timeout_ns=20_000_000, skip_unit=5))
    assert st == mk.MK_OK
    assert mk.mk_status_check(ws) == mk.MK_ERR_TIMEOUT
    C = gu.call_ar(Ad, Bd, mk.MK_F32, ws=ws, opts=ch_opts(tiles))
    gu.assert_bit_exact(gu.host_values(C), oracle.allreduce(A, B))


def test_full_size_every_element_against_the_oracle():
    """The bench workload (P=8, M=N=8192, K_r=3584, random operands, bf16 output) in the default
    (chained) form, compared with the fp64 oracle on every one of its 67 M elements (the oracle
    takes about a minute on the GPU host's cores).  The role split, the unfused baseline and the
    other forms give the same bits (test_full_size_same_bits_as_the_reduce_role), so this covers
    them too."""
    wl = ig.WORKLOADS["ar_mlp_down_p8_m8192_n8192_k3584"]
    A, B, Ad, Bd = gu.upload(wl)
    got = gu.host_values(gu.call_ar(Ad, Bd, mk.MK_BF16, opts=ch_opts()))
    ref = oracle.allreduce(A, B)
    gu.check_tolerance(got, ref, out_bf16=True)


def test_reducescatter_full_size_every_element_against_the_oracle():
    """The ReduceScatter workload (P=8, M=16384, N=8192, K_r=1024, eight 2048-row bf16 shards) in
    the default (chained) form: the shards, concatenated, against the fp64 oracle on every one of
    the 134 M elements (about 40 s of the oracle on the GPU host's cores)."""
    wl = ig.WORKLOADS["rs_p8_m16384_n8192_k1024"]
    A, B, Ad, Bd = gu.upload(wl)
    shards = gu.call_rs(Ad, Bd, mk.MK_BF16, opts=ch_opts())
    got = np.concatenate([gu.host_values(sh) for sh in shards])
    del shards, Ad, Bd
    torch.cuda.empty_cache()
    gu.check_tolerance(got, oracle.allreduce(A, B), out_bf16=True)


def test_reducescatter_full_size_same_bits_and_sampled():
    wl = ig.WORKLOADS["rs_p8_m16384_n8192_k1024"]
    A, B, Ad, Bd = gu.upload(wl)
    want = torch.cat(gu.call_rs(Ad, Bd, mk.MK_BF16), dim=0)          # adaptive role split
    got = torch.cat(gu.call_rs(Ad, Bd, mk.MK_BF16, opts=ch_opts()), dim=0)
    assert torch.equal(got, want)
    rows, cols = gu.sample_indices(wl.M, wl.N, 2048)
    rms = float(np.sqrt(np.mean(oracle.allreduce_rows(A, B, 0, 2) ** 2)))
    gu.check_tolerance(gu.host_values(got)[rows, cols], oracle.allreduce_at(A, B, rows, cols), out_bf16=True,
                       rms_ref=rms)


def test_mid_workload_full_oracle_and_same_bits():
    wl = ig.WORKLOADS["ar_p8_m2048_n4096_k512"]
    A, B, Ad, Bd = gu.upload(wl)
    got = gu.call_ar(Ad, Bd, mk.MK_BF16, opts=ch_opts())
    gu.check_tolerance(gu.host_values(got), oracle.allreduce(A, B), out_bf16=True)
    assert torch.equal(got, gu.call_ar(Ad, Bd, mk.MK_BF16))


@pytest.mark.parametrize("num_ctas", [4, 10, 34])
@pytest.mark.parametrize("M,P", [(256, 4), (256, 8), (1024, 8)])   # tile owners; SM-pair units of all ranks
def test_small_grids(num_ctas, M, P):
    """Few SM pairs, so that every pair claims many tiles (or units) one ahead of the one it
    computes: the result must not depend on the grid."""
    N, Kr = 1024, 128
    wl = ig.Workload("ch_grid", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32", seed=M + num_ctas)
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce(A, B), False)
    C = gu.call_ar(Ad, Bd, mk.MK_F32, opts=ch_opts(num_ctas=num_ctas))
    gu.assert_bit_exact(gu.host_values(C), ref)
