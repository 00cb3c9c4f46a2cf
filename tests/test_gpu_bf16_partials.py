"""bf16 partial tiles (MK_FLAG_BF16_PARTIALS): the compute epilogue rounds each per-rank partial
tile to bf16 before storing it, and the reduce role (or the unfused reduce kernel) widens and
adds them in fp32 in rank order, which is sum_r RNE_bf16(P_r).

On integer inputs every fp32 partial is exact, so its bf16 rounding and the fp32 sum of the
rounded partials are exact too: the result equals the oracle's bf16-partial form bit for bit,
with entries in [-16, 16] so that most partials are large enough to be rounded.  On random
inputs the kernel rounds its fp32 accumulator, the oracle the fp64 value, so a partial may round
to the neighbouring bf16 value where the two straddle a midpoint: at most one bf16 step per
partial, and rarely.
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

INT16 = (ig.DIST_INTEGER, -16.0, 16.0)
MODES = ("adaptive", "static", "unfused")


def bp_opts(mode, tiles="pair", **kw):
    code = {"adaptive": mk.MK_SPLIT_ADAPTIVE, "static": mk.MK_SPLIT_STATIC, "unfused": mk.MK_SPLIT_UNFUSED}[mode]
    fl = kw.pop("flags", 0) | mk.MK_FLAG_BF16_PARTIALS | (mk.MK_FLAG_SINGLE_SM_TILES if tiles == "single" else 0)
    return api.make_opts(code, flags=fl, comm_sms=kw.pop("comm_sms", 4 if mode == "static" else 0), **kw)


SHAPES = [
    # P, M, N, K_r
    (1, 1, 8, 8),
    (2, 128, 256, 64),
    (3, 130, 136, 72),
    (5, 300, 520, 200),
    (16, 64, 256, 64),
    (8, 1100, 1032, 136),
]


@pytest.mark.parametrize("P,M,N,Kr", SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_integer_bit_exact(P, M, N, Kr, out):
    wl = ig.Workload("bp", "allreduce", P, M, N, Kr, INT16, INT16, out, seed=P * 3 + M)
    A, B, Ad, Bd = gu.upload(wl)
    want = oracle.allreduce_bf16_partials(A, B)
    if Kr >= 64:
        assert not np.array_equal(want, oracle.allreduce(A, B))   # partials really are rounded
    ref = gu.rounded_reference(want, out == "bf16")
    code = mk.MK_BF16 if out == "bf16" else mk.MK_F32
    for mode in MODES:
        for tiles in ("pair", "single"):
            C = gu.call_ar(Ad, Bd, code, opts=bp_opts(mode, tiles))
            gu.assert_bit_exact(gu.host_values(C), ref)
    # column slices of the reduction over bf16 tiles (half as many chunks per tile)
    for rs in (2, 8):
        C = gu.call_ar(Ad, Bd, code, opts=bp_opts("adaptive", reduce_split=rs))
        gu.assert_bit_exact(gu.host_values(C), ref)


def test_reducescatter_integer_bit_exact():
    P, M, N, Kr = 4, 1024, 520, 264
    wl = ig.Workload("bp_rs", "reducescatter", P, M, N, Kr, INT16, INT16, "bf16", seed=21)
    A, B, Ad, Bd = gu.upload(wl)
    ref = gu.rounded_reference(oracle.allreduce_bf16_partials(A, B), True)
    for mode in MODES:
        shards = gu.call_rs(Ad, Bd, mk.MK_BF16, opts=bp_opts(mode))
        gu.assert_bit_exact(np.concatenate([gu.host_values(s) for s in shards]), ref)


def _ulp_bf16(x):
    """bf16 spacing at |x| (2^(e-7) for |x| in [2^e, 2^(e+1)))."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


@pytest.mark.parametrize("P,M,N,Kr", [(4, 700, 1032, 512), (8, 384, 768, 1024)])
def test_random_within_one_bf16_step_per_partial(P, M, N, Kr):
    wl = ig.Workload("bp_rnd", "allreduce", P, M, N, Kr, ig.normal(1.0), ig.normal(1.0 / (P * Kr)), "f32", seed=4)
    A, B, Ad, Bd = gu.upload(wl)
    parts = [oracle.gemm(a, b) for a, b in zip(A, B)]
    want = oracle.allreduce_bf16_partials(A, B)
    # one bf16 step per partial that straddles a midpoint, plus the fp32 sum and output rounding
    absq = sum(np.abs(oracle.bf16_to_f64(oracle.round_bf16(p))) for p in parts)
    bound = sum(_ulp_bf16(p) for p in parts) + (P + 1) * 2.0 ** -24 * absq
    outs = {}
    for mode in MODES:
        got = gu.host_values(gu.call_ar(Ad, Bd, mk.MK_F32, opts=bp_opts(mode)))
        err = np.abs(got - want)
        assert (err <= bound).all(), f"{mode}: worst {float((err - bound).max()):.3e} beyond the bound"
        # a flip needs the fp32 accumulator within its own error of a midpoint: rare
        flips = err > (P + 1) * 2.0 ** -24 * absq
        assert flips.mean() < 0.01, f"{mode}: {flips.mean():.4f} of the elements off by a bf16 step"
        # against the exact sum: the relative Frobenius tolerance still holds on the fp32 result,
        # but not the elementwise 1e-2 rms one (P rounded partials can reach 1.07e-2 rms; measured),
        # which is why bf16 partial tiles are an option and not the default
        exact = oracle.allreduce(A, B)
        rel_f = float(np.linalg.norm(got - exact) / np.linalg.norm(exact))
        assert rel_f <= 2e-3, f"{mode}: relative Frobenius error {rel_f:.3e}"
        outs[mode] = got
    # one fixed rank order in every split: the same bits
    assert np.array_equal(outs["adaptive"], outs["unfused"]) and np.array_equal(outs["static"], outs["unfused"])


def test_reducescatter_full_size_sampled():
    wl = ig.WORKLOADS["rs_p8_m16384_n8192_k1024"]
    A, B, Ad, Bd = gu.upload(wl)
    rows, cols = gu.sample_indices(wl.M, wl.N, 4096)
    want = oracle.allreduce_bf16_partials_at(A, B, rows, cols)
    parts = [oracle.allreduce_at([a], [b], rows, cols) for a, b in zip(A, B)]
    absq = sum(np.abs(oracle.bf16_to_f64(oracle.round_bf16(p))) for p in parts)
    step = sum(_ulp_bf16(p) for p in parts) + (wl.P + 1) * 2.0 ** -24 * absq
    for mode in ("adaptive", "unfused"):
        shards = gu.call_rs(Ad, Bd, mk.MK_BF16, opts=bp_opts(mode))
        got = gu.host_values(torch.cat(shards, dim=0))[rows, cols]
        # bf16 output: the bf16 rounding of a value within one bf16 step per partial of the oracle's
        err = np.abs(got - want)
        bound = step + _ulp_bf16(np.maximum(np.abs(got), np.abs(want)))
        assert (err <= bound).all(), f"{mode}: worst {float((err - bound).max()):.3e} beyond the bound"
