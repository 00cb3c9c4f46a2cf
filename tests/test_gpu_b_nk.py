"""MK_FLAG_B_NK: each B[r] given as an N x K_r row-major matrix (K contiguous, the layout of a
linear layer's weight), so that both tensor-core operands are K-major.

The product is the same, so the results must match the oracle exactly on integer inputs in every
split and on both tile kinds, and, on random inputs, must equal the K_r x N layout's result of
the same split bit for bit (the same tile, the same K order).
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
SPLITS = ("adaptive", "static", "unfused", "chained", "accumulate")


def opts(split, tiles, nk, **kw):
    fl = kw.pop("flags", 0) | (mk.MK_FLAG_SINGLE_SM_TILES if tiles == "single" else 0)
    fl |= mk.MK_FLAG_B_NK if nk else 0
    mode = {"adaptive": mk.MK_SPLIT_ADAPTIVE, "static": mk.MK_SPLIT_STATIC, "unfused": mk.MK_SPLIT_UNFUSED,
            "chained": mk.MK_SPLIT_CHAINED, "accumulate": mk.MK_SPLIT_ACCUMULATE}[split]
    return api.make_opts(mode, comm_sms=6 if split == "static" else 0, flags=fl, **kw)


def transposed(Bd):
    return [b.t().contiguous() for b in Bd]


def run(Ad, Bd, out, split, tiles, nk, ws=None, **kw):
    if split == "accumulate" and ws is None:
        ws = api.workspace(mk.MK_OP_ALLREDUCE, len(Ad), Ad[0].shape[0], Bd[0].shape[1], Ad[0].shape[1])
    B = transposed(Bd) if nk else Bd
    # the call takes N from B's second dimension in the K x N layout: pass it explicitly
    P, (M, Kr), N = len(Ad), Ad[0].shape, Bd[0].shape[1]
    dt = torch.bfloat16 if out == mk.MK_BF16 else torch.float32
    C = torch.empty((M, N), dtype=dt, device="cuda")
    if ws is None:
        ws = api.workspace(mk.MK_OP_ALLREDUCE, P, M, N, Kr)
    mk.check(mk.mk_gemm_allreduce(P, M, N, Kr, Ad, B, [C] * P, out, ws, opts=opts(split, tiles, nk, **kw)))
    mk.check(mk.mk_status_check(ws))
    return C


SHAPES = [
    (1, 1, 8, 8),
    (2, 128, 256, 64),
    (3, 130, 136, 72),
    (5, 300, 520, 24),
    (8, 256, 1024, 128),
    (7, 384, 768, 136),
    (4, 1100, 1032, 200),
]


@pytest.mark.parametrize("P,M,N,Kr", SHAPES)
def test_integer_bit_exact_every_split(P, M, N, Kr):
    wl = ig.Workload("bnk", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32", seed=P + M)
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce(A, B), False)
    for tiles in TILES:
        for split in SPLITS:
            C = run(Ad, Bd, mk.MK_F32, split, tiles, True)
            gu.assert_bit_exact(gu.host_values(C), ref)


@pytest.mark.parametrize("P,M,N,Kr", [(2, 128, 256, 64), (5, 300, 520, 24), (8, 256, 1024, 128), (4, 1100, 1032, 200)])
def test_random_same_bits_as_k_by_n(P, M, N, Kr):
    wl = ig.Workload("bnk", "allreduce", P, M, N, Kr, ig.normal(1.0), ig.normal(1.0 / (P * Kr)), "bf16", seed=4)
    A, B, Ad, Bd = gu.upload(wl)
    ref = oracle.allreduce(A, B)
    for tiles in TILES:
        for split in ("adaptive", "unfused", "chained"):
            want = run(Ad, Bd, mk.MK_BF16, split, tiles, False)
            got = run(Ad, Bd, mk.MK_BF16, split, tiles, True)
            gu.check_tolerance(gu.host_values(got), ref, out_bf16=True)
            assert torch.equal(got, want), (split, tiles)


def test_reducescatter():
    P, M, N, Kr = 4, 512, 520, 96
    wl = ig.Workload("bnk_rs", "reducescatter", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "bf16", seed=9)
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce(A, B), True)
    Bt = transposed(Bd)
    for tiles in TILES:
        for split in ("adaptive", "chained"):
            shards = [torch.empty((M // P, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
            ws = api.workspace(mk.MK_OP_REDUCESCATTER, P, M, N, Kr)
            mk.check(mk.mk_gemm_reducescatter(P, M, N, Kr, Ad, Bt, shards, mk.MK_BF16, ws,
                                              opts=opts(split, tiles, True)))
            mk.check(mk.mk_status_check(ws))
            gu.assert_bit_exact(np.concatenate([gu.host_values(s) for s in shards]), ref)


def test_mlp_shape_sampled():
    """The MLP down-projection shape with B given as N x K_r: the chained split equals the
    K_r x N call bit for bit, and sampled elements meet the tolerance against the oracle."""
    wl = ig.WORKLOADS["ar_mlp_down_p8_m8192_n8192_k3584"]
    A, B, Ad, Bd = gu.upload(wl)
    ws = api.workspace(mk.MK_OP_ALLREDUCE, wl.P, wl.M, wl.N, wl.Kr)
    want = run(Ad, Bd, mk.MK_BF16, "chained", "pair", False, ws=ws)
    got = run(Ad, Bd, mk.MK_BF16, "chained", "pair", True, ws=ws)
    assert torch.equal(got, want)
    rows, cols = gu.sample_indices(wl.M, wl.N, 1024)
    rms = float(np.sqrt(np.mean(oracle.allreduce_rows(A, B, 0, 2) ** 2)))
    gu.check_tolerance(gu.host_values(got)[rows, cols], oracle.allreduce_at(A, B, rows, cols), out_bf16=True,
                       rms_ref=rms)
