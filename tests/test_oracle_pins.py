"""Pins for the fp64 oracle against things other than itself.

The pages print no worked numeric example, so the oracle is pinned by: a hand-worked fixture
(tests/golden), exact rational arithmetic on tiny inputs, closed forms, the invariants the
problem fixes (the rank sum equals one GEMM over the concatenated K; rank order does not
matter; ReduceScatter shards concatenate to the AllReduce result), numpy's fp64 matmul as a
special case, torch's fp32->bf16 conversion for the rounding step, and a mutation check that
plants plausible mistakes in a copy of the oracle and shows each one trips a pin.

Problem statement followed: mKernel: Fast Multi-GPU, Multi-Node Fused Kernels, Table 3,
rows GEMM + AllReduce (TP), GEMM + ReduceScatter (TP), AllGather + GEMM (TP).
"""
import ctypes
import json
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import inputgen as ig
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -53


def gamma(n):
    return n * U / (1 - n * U)


def f32_to_bf16_exact(x):
    """Bits of values that are exactly representable in bf16 (asserted)."""
    f = np.asarray(x, np.float32)
    u = f.view(np.uint32)
    assert not (u & 0xFFFF).any(), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def rand_bits(shape, dist, seed, rank, tid):
    a = np.empty(shape, np.uint16)
    ig.fill_bf16(a.reshape(-1), dist, seed, rank, tid)
    return a


def rand_case(P, M, N, Kr, dist_a, dist_b, seed=7):
    A = [rand_bits((M, Kr), dist_a, seed, r, 0) for r in range(P)]
    B = [rand_bits((Kr, N), dist_b, seed, r, 1) for r in range(P)]
    return A, B


def concat(A, B):
    Af = np.concatenate([oracle.bf16_to_f64(a) for a in A], axis=1)
    Bf = np.concatenate([oracle.bf16_to_f64(b) for b in B], axis=0)
    return Af, Bf


# ---------------------------------------------------------------- hand-worked fixture
def test_golden_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "ar_p2_m2_n3_k2_int.json")))
    A = [f32_to_bf16_exact(a) for a in g["A"]]
    B = [f32_to_bf16_exact(b) for b in g["B"]]
    for r in range(g["P"]):
        assert np.array_equal(oracle.gemm(A[r], B[r]), np.array(g["partials"][r], np.float64))
    assert np.array_equal(oracle.allreduce(A, B), np.array(g["C"], np.float64))
    shards = oracle.reducescatter(A, B)
    for s, want in enumerate(g["reducescatter_shards"]):
        assert np.array_equal(shards[s], np.array(want, np.float64))


# ---------------------------------------------------------------- concatenated-K identity
@pytest.mark.parametrize("P,M,N,Kr", [(1, 5, 7, 3), (2, 16, 24, 8), (3, 9, 40, 17), (8, 33, 64, 24),
                                      (16, 4, 8, 2)])
def test_concat_k_identity_integer_exact(P, M, N, Kr):
    A, B = rand_case(P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, seed=P * 100 + M)
    Af, Bf = concat(A, B)
    assert np.array_equal(oracle.allreduce(A, B), Af @ Bf)


@pytest.mark.parametrize("P,M,N,Kr", [(2, 32, 48, 64), (8, 17, 40, 96), (4, 64, 16, 256)])
def test_concat_k_identity_random_within_bound(P, M, N, Kr):
    A, B = rand_case(P, M, N, Kr, ig.normal(1.0), ig.UNIFORM_PM1, seed=11)
    Af, Bf = concat(A, B)
    C = oracle.allreduce(A, B)
    bound = 2 * gamma(P * Kr + P) * (np.abs(Af) @ np.abs(Bf))
    assert (np.abs(C - Af @ Bf) <= bound).all()


# ---------------------------------------------------------------- rank permutation
def test_rank_permutation_invariance():
    P, M, N, Kr = 6, 12, 20, 10
    rng = np.random.default_rng(3)
    perm = rng.permutation(P)
    A, B = rand_case(P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, seed=5)
    C = oracle.allreduce(A, B)
    Cp = oracle.allreduce([A[i] for i in perm], [B[i] for i in perm])
    assert np.array_equal(C, Cp)
    A, B = rand_case(P, M, N, Kr, ig.normal(1.0), ig.normal(0.01), seed=6)
    C = oracle.allreduce(A, B)
    Cp = oracle.allreduce([A[i] for i in perm], [B[i] for i in perm])
    Af, Bf = concat(A, B)
    assert (np.abs(C - Cp) <= 2 * gamma(P * Kr + P) * (np.abs(Af) @ np.abs(Bf))).all()
    # the pairing matters: permuting only the A_r must change the result
    Cx = oracle.allreduce([A[i] for i in perm], B)
    assert not np.allclose(C, Cx)


# ---------------------------------------------------------------- ReduceScatter = AllReduce rows
@pytest.mark.parametrize("P,M", [(2, 8), (4, 12), (8, 16)])
def test_reducescatter_shards_concatenate_to_allreduce(P, M):
    A, B = rand_case(P, M, 24, 16, ig.normal(1.0), ig.normal(1.0), seed=M)
    C = oracle.allreduce(A, B)
    shards = oracle.reducescatter(A, B)
    assert len(shards) == P and all(s.shape == (M // P, 24) for s in shards)
    assert np.array_equal(np.concatenate(shards, axis=0), C)
    A3, B3 = rand_case(3, M + 1 if (M + 1) % 3 else M + 2, 8, 4, ig.normal(1.0), ig.normal(1.0))
    with pytest.raises(ValueError):
        oracle.reducescatter(A3, B3)


# ---------------------------------------------------------------- exact rational brute force
def exact_value(bits):
    return Fraction(float(oracle.bf16_to_f64(np.uint16(bits))))


def exact_round_bf16(x: Fraction) -> int:
    """Round a rational to bf16, nearest-even, by exact integer arithmetic."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    ax = -x if x < 0 else x
    e = ax.numerator.bit_length() - ax.denominator.bit_length()
    if Fraction(2) ** e > ax:
        e -= 1
    while Fraction(2) ** (e + 1) <= ax:
        e += 1
    lead = max(e, -126)
    quantum = Fraction(2) ** (lead - 7)
    q = ax / quantum
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    y = float(n * quantum)
    return sign | int(f32_to_bf16_exact(np.float32(y)))


@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_exact_rationals(seed):
    rng = np.random.default_rng(seed)
    P, M, N, Kr = int(rng.integers(1, 4)), int(rng.integers(1, 9)), int(rng.integers(1, 9)), \
        int(rng.integers(1, 17))
    A, B = rand_case(P, M, N, Kr, ig.normal(1.0), ig.UNIFORM_PM1, seed=100 + seed)
    C = oracle.allreduce(A, B)
    Cb = oracle.round_bf16(C)
    for i in range(M):
        for j in range(N):
            exact = sum((exact_value(A[r][i, k]) * exact_value(B[r][k, j])
                         for r in range(P) for k in range(Kr)), Fraction(0))
            absum = sum((abs(exact_value(A[r][i, k]) * exact_value(B[r][k, j]))
                         for r in range(P) for k in range(Kr)), Fraction(0))
            err = abs(Fraction(C[i, j]) - exact)
            assert err <= Fraction(gamma(P * Kr + P)) * absum
            # the rounded output equals the exact value's rounding unless the exact value sits
            # within the error bound of a rounding midpoint
            want = exact_round_bf16(exact)
            if Cb[i, j] != want:
                lo = exact_round_bf16(exact - Fraction(gamma(P * Kr + P)) * absum)
                hi = exact_round_bf16(exact + Fraction(gamma(P * Kr + P)) * absum)
                assert lo != hi


# ---------------------------------------------------------------- closed forms
def test_closed_form_all_ones():
    P, M, N, Kr = 3, 7, 9, 5
    one = f32_to_bf16_exact(1.0)
    A = [np.full((M, Kr), one, np.uint16) for _ in range(P)]
    B = [np.full((Kr, N), one, np.uint16) for _ in range(P)]
    assert np.array_equal(oracle.allreduce(A, B), np.full((M, N), float(P * Kr)))


def test_closed_form_identity_blocks():
    # A_r = I (K_r = M): C = sum_r B_r
    P, M, N = 4, 6, 10
    eye = f32_to_bf16_exact(np.eye(M, dtype=np.float32))
    A = [eye.copy() for _ in range(P)]
    B = [rand_bits((M, N), ig.INTEGER_PM2, 9, r, 1) for r in range(P)]
    want = sum(oracle.bf16_to_f64(b) for b in B)
    assert np.array_equal(oracle.allreduce(A, B), want)
    # selector: A_r = e_0 e_q^T picks row q of B_r into row 0 (catches an index swap)
    sel = np.zeros((M, M), np.float32)
    sel[0, 3] = 1
    A = [f32_to_bf16_exact(sel)] + [np.zeros((M, M), np.uint16) for _ in range(P - 1)]
    C = oracle.allreduce(A, B)
    assert np.array_equal(C[0], oracle.bf16_to_f64(B[0][3]))
    assert not C[1:].any()


def test_single_rank_is_one_gemm_and_matches_numpy():
    A, B = rand_case(1, 13, 11, 21, ig.INTEGER_PM2, ig.INTEGER_PM2, seed=2)
    C = oracle.allreduce(A, B)
    assert np.array_equal(C, oracle.gemm(A[0], B[0]))
    assert np.array_equal(C, oracle.bf16_to_f64(A[0]) @ oracle.bf16_to_f64(B[0]))


def test_empty_and_degenerate_shapes():
    A, B = rand_case(2, 0, 5, 3, ig.INTEGER_PM2, ig.INTEGER_PM2)
    assert oracle.allreduce(A, B).shape == (0, 5)
    A, B = rand_case(2, 4, 5, 0, ig.INTEGER_PM2, ig.INTEGER_PM2)
    assert np.array_equal(oracle.allreduce(A, B), np.zeros((4, 5)))


def test_sampled_elements_equal_full_result():
    A, B = rand_case(5, 40, 56, 32, ig.normal(1.0), ig.normal(0.5), seed=8)
    C = oracle.allreduce(A, B)
    rng = np.random.default_rng(0)
    rows, cols = rng.integers(0, 40, 300), rng.integers(0, 56, 300)
    assert np.array_equal(oracle.allreduce_at(A, B, rows, cols), C[rows, cols])
    part = oracle.allreduce_rows(A, B, 17, 9)
    assert np.array_equal(part, C[17:26])


def test_allgather_gemm_matches_numpy_blocks():
    P, Mp, K, Np = 4, 3, 12, 5
    As = [rand_bits((Mp, K), ig.INTEGER_PM2, 4, r, 0) for r in range(P)]
    Bs = [rand_bits((K, Np), ig.INTEGER_PM2, 4, r, 1) for r in range(P)]
    Cs = oracle.allgather_gemm(As, Bs)
    Acat = np.concatenate([oracle.bf16_to_f64(a) for a in As], axis=0)
    Bfull = np.concatenate([oracle.bf16_to_f64(b) for b in Bs], axis=1)
    full = Acat @ Bfull
    for r in range(P):
        assert Cs[r].shape == (P * Mp, Np)
        assert np.array_equal(Cs[r], full[:, r * Np:(r + 1) * Np])


# ---------------------------------------------------------------- bf16 partial tiles
def test_bf16_partials_ties_to_even_closed_form():
    # A_r = 1 and B_r[:, j] holding s ones (zeros below) make every partial equal to s.  Between
    # 256 and 512 bf16 steps by 2, so odd s is a tie: 257 -> 256, 259 -> 260, 261 -> 260,
    # 263 -> 264 (even significand); 255 and 256 are exact.  Rounding happens per rank.
    P, M, Kr = 3, 2, 264
    s = [[255, 256, 257, 259, 261, 263],
         [257, 257, 259, 263, 255, 256],
         [263, 261, 255, 257, 259, 257]]
    rounded = {255: 255, 256: 256, 257: 256, 259: 260, 261: 260, 263: 264}
    N = len(s[0])
    one = f32_to_bf16_exact(1.0)
    A = [np.full((M, Kr), one, np.uint16) for _ in range(P)]
    B = []
    for r in range(P):
        b = np.zeros((Kr, N), np.float32)
        for j in range(N):
            b[:s[r][j], j] = 1.0
        B.append(f32_to_bf16_exact(b))
    want = np.array([sum(rounded[s[r][j]] for r in range(P)) for j in range(N)], np.float64)
    got = oracle.allreduce_bf16_partials(A, B)
    assert np.array_equal(got, np.tile(want, (M, 1)))
    # the plain sum is not rounded per rank (column 2: 257 + 259 + 255 = 771, not 256 + 260 + 255)
    assert np.array_equal(oracle.allreduce(A, B)[0], np.array([sum(s[r][j] for r in range(P)) for j in range(N)]))


@pytest.mark.parametrize("Kr", [16, 64])
def test_bf16_partials_equal_the_plain_sum_when_partials_are_exact(Kr):
    # integer entries in {-2..2}: |partial| <= 4 K_r <= 256, every such integer is a bf16 value
    A, B = rand_case(5, 23, 31, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, seed=Kr)
    assert np.array_equal(oracle.allreduce_bf16_partials(A, B), oracle.allreduce(A, B))


def test_bf16_partials_sampled_elements_equal_full_result():
    A, B = rand_case(4, 30, 40, 48, ig.normal(1.0), ig.normal(1.0), seed=12)
    C = oracle.allreduce_bf16_partials(A, B)
    rng = np.random.default_rng(3)
    rows, cols = rng.integers(0, 30, 200), rng.integers(0, 40, 200)
    assert np.array_equal(oracle.allreduce_bf16_partials_at(A, B, rows, cols), C[rows, cols])


@pytest.mark.parametrize("seed", range(4))
def test_bf16_partials_bruteforce_exact_rationals(seed):
    rng = np.random.default_rng(50 + seed)
    P, M, N, Kr = int(rng.integers(1, 4)), int(rng.integers(1, 7)), int(rng.integers(1, 7)), \
        int(rng.integers(1, 17))
    A, B = rand_case(P, M, N, Kr, ig.normal(1.0), ig.UNIFORM_PM1, seed=200 + seed)
    C = oracle.allreduce_bf16_partials(A, B)
    for i in range(M):
        for j in range(N):
            total, absq = Fraction(0), Fraction(0)
            for r in range(P):
                terms = [exact_value(A[r][i, k]) * exact_value(B[r][k, j]) for k in range(Kr)]
                p = sum(terms, Fraction(0))
                bound = Fraction(gamma(Kr)) * sum((abs(t) for t in terms), Fraction(0))
                q = exact_round_bf16(p)
                # a partial within the fp64 error of a rounding midpoint may round either way
                assert q == exact_round_bf16(p - bound) == exact_round_bf16(p + bound), "midpoint case"
                qv = exact_value(q)
                total += qv
                absq += abs(qv)
            assert abs(Fraction(C[i, j]) - total) <= Fraction(gamma(P)) * absq


# ---------------------------------------------------------------- output rounding
def test_round_bf16_hand_cases():
    cases = {
        1.0: 0x3F80, -2.0: 0xC000, 0.0: 0x0000,
        1 + 2 ** -8: 0x3F80,                 # tie -> even (down)
        1 + 3 * 2 ** -8: 0x3F82,             # tie -> even (up)
        1 + 2 ** -8 + 2 ** -30: 0x3F81,      # just above the tie: a detour via fp32 would give 0x3F80
        1 + 2 ** -8 - 2 ** -30: 0x3F80,
        -(1 + 2 ** -7 + 2 ** -9): 0xBF81,
        255.0 * 2 ** 120: 0x7F7F,            # largest finite
        255.5 * 2 ** 120: 0x7F80,            # tie above the largest finite -> even = overflow
        255.4 * 2 ** 120: 0x7F7F,
        2.0 ** -133: 0x0001,                 # smallest subnormal
        2.0 ** -134: 0x0000,                 # half of it: tie -> even (zero)
        3 * 2.0 ** -134: 0x0002,             # 1.5 quanta -> 2
        float("inf"): 0x7F80,
    }
    xs = np.array(list(cases.keys()), np.float64)
    got = oracle.round_bf16(xs)
    for x, g, (k, want) in zip(xs, got, cases.items()):
        assert int(g) == want, (x, hex(int(g)), hex(want))
    assert int(oracle.round_bf16(np.array([np.nan]))[0]) == 0x7FC0
    assert int(oracle.round_bf16(np.array([-0.0]))[0]) == 0x8000


def test_round_bf16_matches_torch_on_fp32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        # exact ties and near-ties around several binades
                        (np.arange(1, 4000, dtype=np.float32) * 2 ** -8 + 1).astype(np.float32),
                        np.float32(rng.uniform(-1e30, 1e30, 1000))])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), want)


def test_round_f32_matches_numpy():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(10000) * 10.0 ** rng.integers(-30, 30, 10000)
    assert np.array_equal(oracle.round_f32(x), x.astype(np.float32))


# ---------------------------------------------------------------- planted mistakes trip a pin
MUTANTS = {
    "drops_last_rank": ("for (int r = 0; r < P; ++r)", "for (int r = 0; r < P - 1; ++r)"),
    "drops_last_k": ("for (int64_t kk = 0; kk < Kr; ++kk)", "for (int64_t kk = 0; kk + 1 < Kr; ++kk)"),
    "subtracts_a_rank": ("c[j] += p[j];", "c[j] += (r == 1 ? -p[j] : p[j]);"),
    "transposes_a": ("bf16_value(A[r][i * Kr + kk])", "bf16_value(A[r][kk * Kr + i])"),
    "transposes_b": ("const uint16_t *b = B[r] + kk * N;\n                    for (int64_t j = 0; j < N; ++j) p[j] += a * bf16_value(b[j]);",
                     "const uint16_t *b = B[r];\n                    for (int64_t j = 0; j < N; ++j) p[j] += a * bf16_value(b[j * N + kk]);"),
    "rounds_ties_away": ("nearbyint(ax / quantum)", "round(ax / quantum)"),
}


def _pins_pass(lib):
    """Run the concatenated-K identity and the tie cases against a (possibly mutated) build."""
    P, M, N, Kr = 3, 8, 8, 8
    A, B = rand_case(P, M, N, Kr, ig.INTEGER_PM2, ig.INTEGER_PM2, seed=21)
    out = np.empty((M, N), np.float64)
    pa = (ctypes.c_void_p * P)(*[a.ctypes.data for a in A])
    pb = (ctypes.c_void_p * P)(*[b.ctypes.data for b in B])
    lib.mko_rank_sum_rows(P, ctypes.c_int64(N), ctypes.c_int64(Kr), pa, pb, ctypes.c_int64(0),
                          ctypes.c_int64(M), out.ctypes.data_as(ctypes.c_void_p))
    Af, Bf = concat(A, B)
    ok_sum = np.array_equal(out, Af @ Bf)
    xs = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 2.0 ** -134], np.float64)
    bits = np.empty(3, np.uint16)
    lib.mko_round_bf16(xs.ctypes.data_as(ctypes.c_void_p), ctypes.c_int64(3),
                       bits.ctypes.data_as(ctypes.c_void_p))
    ok_round = list(bits) == [0x3F80, 0x3F82, 0x0000]
    return ok_sum and ok_round


def _build_variant(tmp_path, name, src):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                           str(so), str(c), "-lm"])
    lib = ctypes.CDLL(str(so))
    lib.mko_rank_sum_rows.restype = None
    lib.mko_round_bf16.restype = None
    return lib


def test_planted_mistakes_are_caught(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mk_oracle.c")).read()
    assert _pins_pass(_build_variant(tmp_path, "unmutated", src))
    for name, (old, new) in MUTANTS.items():
        assert old in src, name
        assert not _pins_pass(_build_variant(tmp_path, name, src.replace(old, new))), name
