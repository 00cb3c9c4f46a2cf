"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small and ragged shapes are compared element by element; the full-size workloads are compared
on sampled elements the oracle computes one by one, plus properties that hold at any size
(fused == unfused bitwise, result independent of the SM split, bf16 output == RNE(fp32
output), ReduceScatter shards == AllReduce rows).
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

MODES = ("adaptive", "static", "unfused")
TILES = ("pair", "single")   # SM-pair 256 x BN tiles (default) or one-SM 128 x BN tiles


def opts_for(mode, comm_sms=4, tiles="pair", **kw):
    if tiles == "single":
        kw["flags"] = kw.get("flags", 0) | mk.MK_FLAG_SINGLE_SM_TILES
    if mode == "adaptive":
        return api.make_opts(mk.MK_SPLIT_ADAPTIVE, **kw)
    if mode == "static":
        return api.make_opts(mk.MK_SPLIT_STATIC, comm_sms=comm_sms, **kw)
    return api.make_opts(mk.MK_SPLIT_UNFUSED, **kw)


def dtype_code(s):
    return mk.MK_BF16 if s == "bf16" else mk.MK_F32


# ------------------------------------------------------------------ the small workload
SMALL = ig.WORKLOADS["ar_p2_m128_n128_k256"]


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("mode", MODES)
def test_small_integer_bit_exact(mode, tiles):
    A, B, Ad, Bd = gu.upload(SMALL, integer=True)
    ref = oracle.allreduce(A, B)
    C = gu.call_ar(Ad, Bd, mk.MK_F32, opts=opts_for(mode, comm_sms=1, tiles=tiles))
    gu.assert_bit_exact(gu.host_values(C), ref)


@pytest.mark.parametrize("tiles", TILES)
@pytest.mark.parametrize("mode", MODES)
def test_small_random_within_tolerance(mode, tiles):
    A, B, Ad, Bd = gu.upload(SMALL)
    ref = oracle.allreduce(A, B)
    C = gu.call_ar(Ad, Bd, mk.MK_F32, opts=opts_for(mode, comm_sms=1, tiles=tiles))
    gu.check_tolerance(gu.host_values(C), ref, out_bf16=False)


# ------------------------------------------------------------------ ragged and edge shapes
EDGE_SHAPES = [
    # P, M, N, K_r
    (1, 1, 8, 8),
    (2, 128, 256, 64),
    (3, 130, 136, 72),      # ragged M, ragged N (BN=256 tile with 136 columns), K below one slice
    (2, 129, 264, 200),     # ragged everything, K not a multiple of 64
    (5, 300, 520, 24),
    (16, 64, 256, 64),      # the most ranks
    (4, 256, 128, 1024),
    (7, 384, 768, 136),
]


@pytest.mark.parametrize("P,M,N,Kr", EDGE_SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_edge_shapes_integer_bit_exact(P, M, N, Kr, out):
    wl = ig.Workload("edge", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, out, seed=P + M)
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce(A, B), out == "bf16")
    for tiles in TILES:
        for mode in MODES:
            C = gu.call_ar(Ad, Bd, dtype_code(out), opts=opts_for(mode, comm_sms=2, tiles=tiles))
            gu.assert_bit_exact(gu.host_values(C), ref)


@pytest.mark.parametrize("P,M,N,Kr", EDGE_SHAPES)
def test_edge_shapes_random_within_tolerance(P, M, N, Kr):
    wl = ig.Workload("edge", "allreduce", P, M, N, Kr, ig.normal(1.0), ig.normal(1.0 / (P * Kr)),
                     "bf16", seed=3)
    A, B, Ad, Bd = gu.upload(wl)
    ref = oracle.allreduce(A, B)
    for tiles in TILES:
        for out in ("f32", "bf16"):
            C = gu.call_ar(Ad, Bd, dtype_code(out), opts=opts_for("adaptive", tiles=tiles))
            gu.check_tolerance(gu.host_values(C), ref, out_bf16=(out == "bf16"))


# Each output tile's reduction cut into column slices claimed as separate items: every element is
# still the rank-ordered sum, so integer inputs stay bit-exact for any slicing, including counts
# that do not divide the tile's chunks (3), the chunk count itself (16), and a clamped request.
@pytest.mark.parametrize("split", [1, 3, 16, 64])
@pytest.mark.parametrize("P,M,N,Kr", [(3, 130, 520, 72), (8, 640, 1032, 128), (12, 256, 264, 64)])
def test_reduce_slices_integer_bit_exact(P, M, N, Kr, split):
    wl = ig.Workload("slices", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32", seed=split)
    A, B, Ad, Bd = gu.upload(wl)
    ref = oracle.allreduce(A, B)
    for tiles in TILES:
        for mode in MODES:
            C = gu.call_ar(Ad, Bd, mk.MK_F32, opts=opts_for(mode, comm_sms=2, tiles=tiles, reduce_split=split))
            gu.assert_bit_exact(gu.host_values(C), ref)
    if M % P == 0:
        for mode in MODES:
            out = gu.call_rs(Ad, Bd, mk.MK_F32, opts=opts_for(mode, comm_sms=2, reduce_split=split))
            gu.assert_bit_exact(np.concatenate([gu.host_values(x) for x in out]), ref)


# Both compute orders (bands of tile rows rank by rank, the default, or the P ranks of each tile
# back to back) and band heights that leave a short last band must give the same bits.
@pytest.mark.parametrize("order", ["rank_major", "tile_major"])
@pytest.mark.parametrize("band", [0, 1, 3])
def test_compute_orders_integer_bit_exact(order, band):
    P, M, N, Kr = 6, 1400, 776, 136
    wl = ig.Workload("order", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32", seed=band)
    A, B, Ad, Bd = gu.upload(wl)
    ref = oracle.allreduce(A, B)
    fl = mk.MK_FLAG_TILE_MAJOR if order == "tile_major" else mk.MK_FLAG_RANK_MAJOR
    for tiles in TILES:
        for mode in MODES:
            C = gu.call_ar(Ad, Bd, mk.MK_F32, opts=opts_for(mode, comm_sms=6, tiles=tiles, flags=fl, raster_group=band))
            gu.assert_bit_exact(gu.host_values(C), ref)


def test_zero_k_gives_zeros_and_empty_is_noop():
    P, M, N = 3, 200, 136
    Ad = [torch.empty((M, 0), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    Bd = [torch.empty((0, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    C = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    gu.call_ar(Ad, Bd, mk.MK_F32, C=C)
    assert not C.any()
    Ad = [torch.empty((0, 64), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    Bd = [torch.zeros((64, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    C = gu.call_ar(Ad, Bd, mk.MK_F32)
    assert C.shape == (0, N)


def test_distinct_output_buffers_all_receive_the_result():
    wl = ig.Workload("bcast", "allreduce", 4, 256, 512, 128, ig.INTEGER_PM2, ig.INTEGER_PM2, "bf16")
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce(A, B), True)
    Cs = [torch.empty((256, 512), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    gu.call_ar(Ad, Bd, mk.MK_BF16, C=Cs)
    for c in Cs:
        gu.assert_bit_exact(gu.host_values(c), ref)


def test_reducescatter_small_and_ragged_shards():
    for P, M, N, Kr in [(2, 256, 256, 64), (3, 192, 136, 40), (8, 1024, 512, 64)]:
        wl = ig.Workload("rs", "reducescatter", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "bf16")
        A, B, Ad, Bd = gu.upload(wl)
        want = [gu.rounded_reference(s, True) for s in oracle.reducescatter(A, B)]
        for tiles in TILES:
            for mode in MODES:
                shards = gu.call_rs(Ad, Bd, mk.MK_BF16, opts=opts_for(mode, comm_sms=2, tiles=tiles))
                for s in range(P):
                    gu.assert_bit_exact(gu.host_values(shards[s]), want[s])


def test_workspace_reuse_across_calls_and_shapes():
    ws = api.workspace(mk.MK_OP_ALLREDUCE, 8, 512, 1024, 256)
    for i, (P, M, N, Kr) in enumerate([(8, 512, 1024, 256), (4, 256, 512, 128), (8, 512, 1024, 256),
                                       (2, 128, 256, 64)]):
        wl = ig.Workload("reuse", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32",
                         seed=i)
        A, B, Ad, Bd = gu.upload(wl)
        for tiles in TILES:
            for mode in MODES:
                C = gu.call_ar(Ad, Bd, mk.MK_F32, opts=opts_for(mode, tiles=tiles), ws=ws)
                gu.assert_bit_exact(gu.host_values(C), oracle.allreduce(A, B))


# ------------------------------------------------------------------ the 2048 x 4096 workload
MID = ig.WORKLOADS["ar_p8_m2048_n4096_k512"]


def test_mid_workload_full_oracle_comparison():
    A, B, Ad, Bd = gu.upload(MID)
    ref = oracle.allreduce(A, B)
    outs = {}
    for mode in MODES:
        outs[mode] = gu.call_ar(Ad, Bd, mk.MK_BF16, opts=opts_for(mode, comm_sms=16))
        gu.check_tolerance(gu.host_values(outs[mode]), ref, out_bf16=True)
    c32 = gu.call_ar(Ad, Bd, mk.MK_F32)
    gu.check_tolerance(gu.host_values(c32), ref, out_bf16=False)
    single = gu.call_ar(Ad, Bd, mk.MK_BF16, opts=opts_for("adaptive", tiles="single"))
    gu.check_tolerance(gu.host_values(single), ref, out_bf16=True)
    # one fixed-order sum regardless of the schedule, and bf16 = RNE(fp32) of that sum
    assert torch.equal(outs["adaptive"], outs["unfused"]) and torch.equal(outs["static"], outs["unfused"])
    assert torch.equal(outs["adaptive"], c32.to(torch.bfloat16))


def test_mid_workload_integer_bit_exact():
    A, B, Ad, Bd = gu.upload(MID, integer=True)
    ref = gu.rounded_reference(oracle.allreduce(A, B), True)
    C = gu.call_ar(Ad, Bd, mk.MK_BF16)
    gu.assert_bit_exact(gu.host_values(C), ref)


# ------------------------------------------------------------------ full-size workloads (sampled)
def sampled_check(wl, out_tensor_fn, integer=False, n=4096):
    A, B, Ad, Bd = gu.upload(wl, integer=integer)
    rows, cols = gu.sample_indices(wl.M, wl.N, n)
    ref = oracle.allreduce_at(A, B, rows, cols)
    out = out_tensor_fn(Ad, Bd)
    got = gu.host_values(out)[rows, cols]
    if integer:
        gu.assert_bit_exact(got, gu.rounded_reference(ref, True))
    else:
        # rms of the full C from a row sample of the oracle (the sampled elements are random)
        rms_rows = oracle.allreduce_rows(A, B, 0, 2)
        gu.check_tolerance(got, ref, out_bf16=True, rms_ref=float(np.sqrt(np.mean(rms_rows ** 2))))
    return Ad, Bd, out


MLP = ig.WORKLOADS["ar_mlp_down_p8_m8192_n8192_k3584"]


def test_mlp_down_projection_sampled_and_schedule_invariant():
    Ad, Bd, C = sampled_check(MLP, lambda Ad, Bd: gu.call_ar(Ad, Bd, mk.MK_BF16))
    for mode, nr in (("unfused", 0), ("static", 2), ("static", 16), ("static", gu.num_sms() // 2)):
        other = gu.call_ar(Ad, Bd, mk.MK_BF16, opts=opts_for(mode, comm_sms=nr))
        assert torch.equal(C, other), (mode, nr)


def test_mlp_down_projection_integer_sampled_bit_exact():
    sampled_check(MLP, lambda Ad, Bd: gu.call_ar(Ad, Bd, mk.MK_BF16), integer=True)


RS = ig.WORKLOADS["rs_p8_m16384_n8192_k1024"]


def test_reducescatter_full_size_sampled_and_equal_to_allreduce_rows():
    shards_box = {}

    def run(Ad, Bd):
        shards_box["s"] = gu.call_rs(Ad, Bd, mk.MK_BF16)
        return torch.cat(shards_box["s"], dim=0)

    Ad, Bd, cat = sampled_check(RS, run)
    ar = gu.call_ar(Ad, Bd, mk.MK_BF16)
    assert torch.equal(cat, ar)
    assert all(s.shape == (RS.M // RS.P, RS.N) for s in shards_box["s"])


@pytest.mark.parametrize("M", ig.SWEEP_M)
def test_sweep_shapes_sampled_and_split_invariant(M):
    wl = ig.sweep_workload(M)
    Ad, Bd, C = sampled_check(wl, lambda Ad, Bd: gu.call_ar(Ad, Bd, mk.MK_BF16), n=1024)
    for nr in (2, gu.num_sms() - 2):
        assert torch.equal(C, gu.call_ar(Ad, Bd, mk.MK_BF16, opts=opts_for("static", comm_sms=nr)))
    assert torch.equal(C, gu.call_ar(Ad, Bd, mk.MK_BF16, opts=opts_for("unfused")))
