"""Ring Attention (sequence parallelism) through the C ABI against the fp64 oracle.

mKernel: Fast Multi-GPU, Multi-Node Fused Kernels, Table 3, row "Ring Attention (SP)": each rank's
queries attend to every rank's KV slice, visited in ring order; communication blocks forward the
KV tiles to the next rank and release a flag per 128-row tile, compute blocks acquire it.

Tolerance, derived from the arithmetic.  Scores are fp32 sums of exact bf16 products; the
probabilities p = 2^(s * scale * log2 e - m) are rounded to bf16 before P V, which multiplies each
probability by (1 + delta) with |delta| <= 2^-9; the row sum and every accumulation stay fp32.  The
rounding of the probabilities then adds to O[i][c] an error of standard deviation 2^-9 / sqrt(3)
times e[i][c] = sqrt(sum_j w_j^2 V[j][c]^2) / l, which the oracle returns.  Every element must lie
within eight standard deviations of it (plus 1e-6 for the fp32 arithmetic the model leaves out,
and half a bf16 ulp for bf16 outputs), and the relative Frobenius error must stay within 3e-3.
Exact cases (all-zero queries: the mean of V; one dominant key: that key's value row) are compared
bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gemm_tile_level_gb300 import api, mk
    import gpu_util as gu

SIGMA = 2.0 ** -9 / math.sqrt(3.0)


def upload(Q, K, V):
    return ([api.bf16_device(q) for q in Q], [api.bf16_device(k) for k in K], [api.bf16_device(v) for v in V])


def run(Qd, Kd, Vd, out=None, split="fused", ring=True, scale=0.0, comm_sms=0, ws=None):
    out = mk.MK_BF16 if out is None else out
    mode = {"fused": mk.MK_SPLIT_ADAPTIVE, "static": mk.MK_SPLIT_STATIC, "unfused": mk.MK_SPLIT_UNFUSED}[split]
    opts = api.make_opts(mode, comm_sms=comm_sms)
    O, L, R, st = api.ring_attention(Qd, Kd, Vd, out, scale=scale, ring=ring, ws=ws, opts=opts)
    mk.check(st)
    torch.cuda.synchronize()
    return O, L, R


def values(t):
    return gu.host_values(t)


def check_against_oracle(O_gpu, L_gpu, ref, out_bf16, lse_check=True):
    """O_gpu, L_gpu: lists over ranks of device tensors; ref: (O, L, E) lists of fp64 arrays."""
    O_ref, L_ref, E_ref = ref
    num = den = 0.0
    for r in range(len(O_gpu)):
        got = values(O_gpu[r])
        want = O_ref[r]
        err = np.abs(got - want)
        bound = 8 * SIGMA * E_ref[r] + 1e-6
        if out_bf16:
            bound = bound + gu.ulp_bf16(want) / 2
        bad = err > bound
        assert not bad.any(), (f"rank {r}: {int(bad.sum())} elements beyond the bound; worst excess "
                               f"{(err - bound).max():.3e} at {np.argwhere(bad)[0]}")
        num += float(((got - want) ** 2).sum())
        den += float((want ** 2).sum())
        if lse_check and L_gpu is not None:
            lg = L_gpu[r].cpu().numpy().astype(np.float64)
            assert np.abs(lg - L_ref[r]).max() <= 1e-5 * np.abs(L_ref[r]).max() + 1e-5
    rel = math.sqrt(num / den)
    assert rel <= 3e-3, f"relative Frobenius error {rel:.3e}"
    return rel


SHAPES = [
    # P, H, S
    (2, 2, 256),
    (1, 3, 128),
    (3, 1, 200),     # ragged KV and query tiles
    (4, 2, 384),     # one and a half query units per slice
    (2, 1, 64),
    (8, 2, 128),
    (16, 1, 256),    # the most ranks: fifteen forwarding steps
    (5, 2, 640),     # odd P, a unit and a quarter per slice, ragged last KV tile of 128
]


@pytest.mark.parametrize("P,H,S", SHAPES)
@pytest.mark.parametrize("split", ["fused", "unfused"])
def test_random_within_tolerance_and_forms_agree(P, H, S, split):
    wl = ig.AttnWorkload("t", P, H, S, 128, ig.normal(1.0), ig.normal(1.0), ig.normal(1.0), seed=P * 1000 + S)
    Q, K, V = ig.make_attn_operands(wl)
    Qd, Kd, Vd = upload(Q, K, V)
    ref = oracle.ring_attention(Q, K, V)
    O32, L32, R = run(Qd, Kd, Vd, mk.MK_F32, split=split)
    check_against_oracle(O32, L32, ref, out_bf16=False)
    O16, L16, _ = run(Qd, Kd, Vd, mk.MK_BF16, split=split)
    check_against_oracle(O16, L16, ref, out_bf16=True)
    # the bf16 output is the fp32 result rounded to nearest even, bit for bit
    for r in range(P):
        assert torch.equal(O16[r], O32[r].to(torch.bfloat16))
        assert torch.equal(L16[r], L32[r])
    # reading every slice in place gives the same bits as reading the forwarded copies
    Oi, Li, _ = run(Qd, Kd, Vd, mk.MK_F32, ring=False)
    for r in range(P):
        assert torch.equal(Oi[r], O32[r]) and torch.equal(Li[r], L32[r])
    # the ring buffers hold the forwarded slices: slot s-1 of rank r is the KV of rank (r - s) mod P
    if P > 1:
        for r in range(P):
            for s in range(1, P):
                o = (r - s) % P
                assert torch.equal(R[r][s - 1, 0], Kd[o]) and torch.equal(R[r][s - 1, 1], Vd[o]), (r, s)


@pytest.mark.parametrize("comm_sms", [1, 3, 40])
def test_static_copy_split_gives_the_same_bits(comm_sms):
    wl = ig.AttnWorkload("t", 4, 3, 256, 128, ig.normal(1.0), ig.normal(1.0), ig.normal(1.0), seed=7)
    Q, K, V = ig.make_attn_operands(wl)
    Qd, Kd, Vd = upload(Q, K, V)
    O, L, _ = run(Qd, Kd, Vd, mk.MK_F32)
    O2, L2, _ = run(Qd, Kd, Vd, mk.MK_F32, split="static", comm_sms=comm_sms)
    for r in range(4):
        assert torch.equal(O[r], O2[r]) and torch.equal(L[r], L2[r])


def test_zero_queries_give_the_mean_of_v_bit_exact():
    # scores all 0: every probability is 2^0 = 1 exactly, the sums of integer values are exact in
    # fp32 and the division by the number of keys (a power of two) is exact
    P, H, S, d = 4, 2, 256, 128
    rng = np.random.default_rng(1)
    Q = [np.zeros((H, S, d), np.uint16) for _ in range(P)]
    K = [oracle.round_bf16(rng.standard_normal((H, S, d))) for _ in range(P)]
    V = [oracle.round_bf16(rng.integers(-2, 3, (H, S, d)).astype(np.float64)) for _ in range(P)]
    Qd, Kd, Vd = upload(Q, K, V)
    ref = oracle.ring_attention(Q, K, V)
    for split in ("fused", "unfused"):
        O, L, _ = run(Qd, Kd, Vd, mk.MK_F32, split=split)
        for r in range(P):
            gu.assert_bit_exact(values(O[r]), ref[0][r])
            assert np.allclose(L[r].cpu().numpy(), math.log(P * S), rtol=1e-6, atol=0)


def test_one_dominant_key_returns_its_value_row_bit_exact():
    # with scale = ln 2 the log2-domain scale is 1, so the winning key's probability is 2^0 = 1
    # exactly and every other key's is 2^-2048 = 0
    P, H, S, d = 4, 2, 256, 128
    rng = np.random.default_rng(2)
    Q = [np.zeros((H, S, d)) for _ in range(P)]
    K = [np.zeros((H, S, d)) for _ in range(P)]
    V = [rng.integers(-8, 9, (H, S, d)).astype(np.float64) for _ in range(P)]
    targets = {}
    for h in range(H):
        for r in range(P):
            for i in range(0, S, 7):
                c = int(rng.integers(d))
                o, j = int(rng.integers(P)), int(rng.integers(S))
                if K[o][h, j].any():
                    continue
                Q[r][h, i, c] = 2048.0
                K[o][h, j, c] = 1.0
                targets[(r, h, i)] = (o, j, c)
    # a query whose direction another target key also uses would see two winners: keep one per direction
    Qb = [oracle.round_bf16(x) for x in Q]
    Kb = [oracle.round_bf16(x) for x in K]
    Vb = [oracle.round_bf16(x) for x in V]
    Qd, Kd, Vd = upload(Qb, Kb, Vb)
    scale = float(np.float32(math.log(2.0)))
    O, _, _ = run(Qd, Kd, Vd, mk.MK_F32, scale=scale)
    ref = oracle.ring_attention(Qb, Kb, Vb, scale=scale)
    checked = 0
    for (r, h, i), (o, j, c) in targets.items():
        # only rows whose direction is unique among the target keys have a single winner
        want = ref[0][r][h, i]
        if np.array_equal(want, V[o][h, j]):
            assert np.array_equal(values(O[r])[h, i], V[o][h, j]), (r, h, i)
            checked += 1
    assert checked > 50


def test_growing_scores_raise_the_maximum_inside_tiles():
    """Scores that rise by more than 2^8 every 16 keys: every chunk of every tile raises a row's
    running maximum, so the probabilities already formed (stored in TMEM or still in registers)
    and their sum are rescaled; within tolerance of the oracle, and the in-place form agrees."""
    P, H, S, d = 2, 2, 256, 128
    rng = np.random.default_rng(11)
    Q = [np.zeros((H, S, d)) for _ in range(P)]
    K = [np.zeros((H, S, d)) for _ in range(P)]
    V = [rng.standard_normal((H, S, d)) for _ in range(P)]
    for r in range(P):
        Q[r][:, :, 0] = 4.0
        Q[r][:, :, 1] = rng.uniform(-1, 1, (H, S))
        # s * scale * log2(e) rises by about 0.7 per key: more than 8 per 16-key chunk
        K[r][:, :, 0] = np.arange(r * S, (r + 1) * S) * 1.4
        K[r][:, :, 1] = rng.uniform(-1, 1, (H, S))
    Qb = [oracle.round_bf16(x) for x in Q]
    Kb = [oracle.round_bf16(x) for x in K]
    Vb = [oracle.round_bf16(x) for x in V]
    Qd, Kd, Vd = upload(Qb, Kb, Vb)
    ref = oracle.ring_attention(Qb, Kb, Vb)
    for split in ("fused", "unfused"):
        O32, L32, _ = run(Qd, Kd, Vd, mk.MK_F32, split=split)
        check_against_oracle(O32, L32, ref, out_bf16=False)
    Oi, Li, _ = run(Qd, Kd, Vd, mk.MK_F32, ring=False)
    for r in range(P):
        assert torch.equal(Oi[r], O32[r]) and torch.equal(Li[r], L32[r])


def test_full_size_workload_sampled():
    """The bench workload (8 ranks x 4096 tokens, 32 heads of 128): sampled query rows of every
    rank against the oracle, and the in-place and forwarded forms bit for bit."""
    wl = ig.ATTN_WORKLOADS["ring_p8_h32_s4096_d128"]
    Q, K, V = ig.make_attn_operands(wl)
    Qd, Kd, Vd = upload(Q, K, V)
    O, L, _ = run(Qd, Kd, Vd, mk.MK_BF16)
    O2, L2, _ = run(Qd, Kd, Vd, mk.MK_BF16, ring=False)
    rng = np.random.default_rng(3)
    num = den = 0.0
    for r in range(wl.P):
        assert torch.equal(O[r], O2[r]) and torch.equal(L[r], L2[r])
        for h in rng.choice(wl.H, 2, replace=False):
            rows = np.sort(rng.choice(wl.S, 6, replace=False))
            rows[0] = 0
            o, l, e = oracle.attention_rows(Q, K, V, r, int(h), rows)
            got = values(O[r][int(h)])[rows]
            bound = 8 * SIGMA * e + 1e-6 + gu.ulp_bf16(o) / 2
            assert (np.abs(got - o) <= bound).all(), (r, h)
            assert np.abs(L[r][int(h)].cpu().numpy()[rows] - l).max() <= 1e-4
            num += float(((got - o) ** 2).sum())
            den += float((o ** 2).sum())
    assert math.sqrt(num / den) <= 3e-3


def test_a_withheld_tile_times_out_and_the_next_call_recovers():
    """Fault injection on the host side: one forwarded KV tile is never copied, so the compute that
    needs it waits out its (short) limit; the call reports MK_ERR_TIMEOUT through the workspace and
    exits cleanly, and the next call on the same workspace is correct."""
    wl = ig.AttnWorkload("t", 4, 2, 256, 128, ig.normal(1.0), ig.normal(1.0), ig.normal(1.0), seed=3)
    Q, K, V = ig.make_attn_operands(wl)
    Qd, Kd, Vd = upload(Q, K, V)
    ws = api.ring_attention_workspace(4, 2, 256, 128)
    want, _, _ = run(Qd, Kd, Vd, mk.MK_F32)
    opts = api.make_opts(mk.MK_SPLIT_ADAPTIVE, timeout_ns=50_000_000, skip_unit=5)
    _, _, _, st = api.ring_attention(Qd, Kd, Vd, mk.MK_F32, ws=ws, opts=opts)
    mk.check(st)
    assert mk.mk_status_check(ws) == mk.MK_ERR_TIMEOUT
    assert mk.mk_status_check(ws) == mk.MK_OK   # read and cleared
    got, _, _ = run(Qd, Kd, Vd, mk.MK_F32, ws=ws)
    for r in range(4):
        assert torch.equal(got[r], want[r])
