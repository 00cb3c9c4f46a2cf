"""Epilogue pacing: the epilogue may pause between its 32-column store chunks (on by default for
the unfused and role-split modes, and for chained and accumulate modes when K_r >= 2048).
Pacing moves stores in time only, so every mode must give the oracle's values on integer inputs
and, on random inputs, the same bits with and without MK_FLAG_NO_EPILOGUE_PACING.
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

MODES = ("unfused", "adaptive", "static", "chained", "accumulate")
# K_r = 2104 is 33 k-blocks (the last one ragged): paced in every mode
SHAPES = [(3, 300, 520, 2104), (8, 640, 1024, 2048)]


def _opts(mode, paced, tiles="pair"):
    code = {"unfused": mk.MK_SPLIT_UNFUSED, "adaptive": mk.MK_SPLIT_ADAPTIVE, "static": mk.MK_SPLIT_STATIC,
            "chained": mk.MK_SPLIT_CHAINED, "accumulate": mk.MK_SPLIT_ACCUMULATE}[mode]
    fl = (0 if paced else mk.MK_FLAG_NO_EPILOGUE_PACING) | (mk.MK_FLAG_SINGLE_SM_TILES if tiles == "single" else 0)
    return api.make_opts(code, flags=fl, comm_sms=4 if mode == "static" else 0)


@pytest.mark.parametrize("P,M,N,Kr", SHAPES)
@pytest.mark.parametrize("mode", MODES)
def test_integer_bit_exact_paced_and_unpaced(P, M, N, Kr, mode):
    wl = ig.Workload("pace", "allreduce", P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32", seed=P + M)
    A, B, Ad, Bd = gu.upload(wl)
    ref = oracle.allreduce(A, B)
    for tiles in ("pair", "single"):
        for paced in (True, False):
            C = gu.call_ar(Ad, Bd, mk.MK_F32, opts=_opts(mode, paced, tiles))
            gu.assert_bit_exact(gu.host_values(C), ref)


@pytest.mark.parametrize("mode", ("unfused", "adaptive", "static", "chained"))
def test_random_same_bits_paced_and_unpaced(mode):
    P, M, N, Kr = 4, 700, 1032, 2304
    wl = ig.Workload("pace_rnd", "allreduce", P, M, N, Kr, ig.normal(1.0), ig.normal(1.0 / (P * Kr)), "bf16", seed=8)
    A, B, Ad, Bd = gu.upload(wl)
    paced = gu.call_ar(Ad, Bd, mk.MK_BF16, opts=_opts(mode, True))
    gu.check_tolerance(gu.host_values(paced), oracle.allreduce(A, B), out_bf16=True)
    assert torch.equal(paced, gu.call_ar(Ad, Bd, mk.MK_BF16, opts=_opts(mode, False)))
    # and the same bits as the unfused baseline (the fixed rank order of every mode but accumulate)
    assert torch.equal(paced, gu.call_ar(Ad, Bd, mk.MK_BF16, opts=_opts("unfused", True)))


def test_allgather_same_bits_paced_and_unpaced():
    P, M, N, K = 4, 1024, 520, 2048
    A = [np.empty((M // P, K), np.uint16) for _ in range(P)]
    B = [np.empty((K, N), np.uint16) for _ in range(P)]
    for r in range(P):
        ig.fill_bf16(A[r].reshape(-1), ig.normal(1.0), 3, r, ig.TID_A)
        ig.fill_bf16(B[r].reshape(-1), ig.normal(1.0 / K), 3, r, ig.TID_B)
    Ad = [api.bf16_device(a) for a in A]
    Bd = [api.bf16_device(b) for b in B]
    outs = []
    for fl in (0, mk.MK_FLAG_NO_EPILOGUE_PACING):
        ws = api.workspace(mk.MK_OP_ALLGATHER_GEMM, P, M, N, K)
        C, _, st = api.allgather_gemm(Ad, Bd, mk.MK_F32, ws=ws, opts=api.make_opts(mk.MK_SPLIT_ADAPTIVE, flags=fl))
        mk.check(st)
        mk.check(mk.mk_status_check(ws))
        outs.append(C)
    want = oracle.allgather_gemm(A, B)
    for r in range(P):
        gu.check_tolerance(gu.host_values(outs[0][r]), want[r], out_bf16=False)
        assert torch.equal(outs[0][r], outs[1][r])
