"""Pins of the Ring Attention oracle (oracle/mk_oracle_attn.c) to things other than itself.

mKernel: Fast Multi-GPU, Multi-Node Fused Kernels, Table 3, row "Ring Attention (SP)": every
rank's queries attend to the keys and values of the whole sequence, whose slices the ring brings
to each rank in turn.  The oracle is softmax attention written out in fp64.  It is pinned by:
  * closed forms: all-zero queries give the mean of V and lse = log(#keys) exactly; one dominant
    key returns that key's value row exactly; two keys give the logistic weighting of their
    values (which fixes the scale factor and which operand the scores use);
  * invariants: the order of the KV slices (which rank's slice comes first on the ring) changes
    nothing but rounding; adding one vector to every key shifts every score of a query by the
    same amount and leaves O unchanged; values of ones give ones;
  * library routines: numpy's fp64 exp and matmul give the same result on random inputs;
  * a 50-digit brute force (mpmath) on tiny inputs, for O, lse and the error scale;
  * planted mistakes in a copy of the oracle, each of which trips one of the pins above.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import inputgen as ig
import oracle


def bits(x):
    """fp64 values exactly representable in bf16 -> bf16 bit patterns."""
    b = oracle.round_bf16(np.asarray(x, np.float64))
    assert np.array_equal(oracle.bf16_to_f64(b), np.asarray(x, np.float64)), "value not exact in bf16"
    return b


def rand_bits(shape, rng, scale=1.0):
    return oracle.round_bf16(rng.standard_normal(shape) * scale)


def full(Q, K, V, rows_fn=None, scale=None):
    """Every rank's O and lse through `rows_fn` (the oracle's attention_rows by default)."""
    rows_fn = rows_fn or oracle.attention_rows
    P = len(Q)
    H, S, d = Q[0].shape
    O = np.empty((P, H, S, d))
    L = np.empty((P, H, S))
    E = np.empty((P, H, S, d))
    for r in range(P):
        for h in range(H):
            O[r, h], L[r, h], E[r, h] = rows_fn(Q, K, V, r, h, np.arange(S), scale)
    return O, L, E


def numpy_attention(Q, K, V, scale=None):
    P = len(Q)
    H, S, d = Q[0].shape
    scale = 1 / np.sqrt(d) if scale is None else scale
    Kc = np.concatenate([oracle.bf16_to_f64(k) for k in K], axis=1)   # H x PS x d
    Vc = np.concatenate([oracle.bf16_to_f64(v) for v in V], axis=1)
    O = np.empty((P, H, S, d))
    L = np.empty((P, H, S))
    for r in range(P):
        q = oracle.bf16_to_f64(Q[r])
        for h in range(H):
            s = q[h] @ Kc[h].T * scale
            m = s.max(axis=1, keepdims=True)
            w = np.exp(s - m)
            O[r, h] = (w @ Vc[h]) / w.sum(axis=1, keepdims=True)
            L[r, h] = m[:, 0] + np.log(w.sum(axis=1))
    return O, L


# ---------------------------------------------------------------- closed forms
def test_zero_queries_give_the_mean_of_v_exactly():
    rng = np.random.default_rng(0)
    P, H, S, d = 3, 2, 64, 16
    Q = [bits(np.zeros((H, S, d))) for _ in range(P)]
    K = [rand_bits((H, S, d), rng) for _ in range(P)]
    V = [bits(rng.integers(-2, 3, (H, S, d)).astype(np.float64)) for _ in range(P)]
    O, L, E = full(Q, K, V)
    Vc = np.concatenate([oracle.bf16_to_f64(v) for v in V], axis=1)
    mean = Vc.sum(axis=1) / (P * S)                      # integer sum: exact; one rounding
    for r in range(P):
        for h in range(H):
            assert np.array_equal(O[r, h], np.broadcast_to(mean[h], (S, d)))
            assert np.all(L[r, h] == np.log(P * S))
            assert np.allclose(E[r, h], np.sqrt((Vc[h] ** 2).sum(axis=0)) / (P * S), rtol=1e-15, atol=0)


def test_one_dominant_key_returns_its_value_row_exactly():
    rng = np.random.default_rng(1)
    P, H, S, d = 3, 2, 32, 16
    alpha = 2048.0                                       # scale 1/4: winning score 512, others 0
    Q = [np.zeros((H, S, d)) for _ in range(P)]
    K = [np.zeros((H, S, d)) for _ in range(P)]
    # nonzero values: the other keys still add exp(-512) * v (about 1e-222 * v), far below half an
    # ulp of any nonzero v, so the winning row comes back exactly
    V = [(rng.integers(1, 9, (H, S, d)) * rng.choice([-1, 1], (H, S, d))).astype(np.float64) for _ in range(P)]
    targets = {}
    for h in range(H):
        used = set()
        for c in range(d):                               # query rows 0..d-1 of rank c % P, direction c
            r, i = c % P, c // P
            o, j = int(rng.integers(P)), int(rng.integers(S))
            while (o, j) in used:
                o, j = int(rng.integers(P)), int(rng.integers(S))
            used.add((o, j))
            Q[r][h, i, c] = alpha
            K[o][h, j, c] = 1.0
            targets[(r, h, i)] = (o, j)
    Qb, Kb, Vb = [bits(x) for x in Q], [bits(x) for x in K], [bits(x) for x in V]
    O, L, _ = full(Qb, Kb, Vb)
    for (r, h, i), (o, j) in targets.items():
        assert np.array_equal(O[r, h, i], V[o][h, j]), (r, h, i)
        assert L[r, h, i] == 512.0


def test_two_keys_give_the_logistic_weighting():
    P, H, S, d = 2, 1, 1, 4
    for a in (-3.0, 0.5, 2.0, 7.0):
        Q = [bits(np.array([[[a, 0, 0, 0]]])), bits(np.array([[[0, a, 0, 0]]]))]
        K = [bits(np.array([[[1.0, 0, 0, 0]]])), bits(np.zeros((1, 1, 4)))]
        V = [bits(np.array([[[1.0, 2.0, -4.0, 0.5]]])), bits(np.array([[[-1.0, 0.25, 8.0, 3.0]]]))]
        O, L, _ = full(Q, K, V)
        s0 = a * 0.5                                      # scale 1/sqrt(4)
        w0 = np.exp(s0 - max(s0, 0.0))
        w1 = np.exp(0.0 - max(s0, 0.0))
        want = (w0 * oracle.bf16_to_f64(V[0][0, 0]) + w1 * oracle.bf16_to_f64(V[1][0, 0])) / (w0 + w1)
        assert np.allclose(O[0, 0, 0], want, rtol=1e-15, atol=1e-15)
        assert abs(L[0, 0, 0] - (max(s0, 0.0) + np.log(w0 + w1))) <= 1e-15 * max(1.0, abs(L[0, 0, 0]))
        # rank 1's query points along column 1, where both keys are zero: equal weights
        assert np.allclose(O[1, 0, 0], (oracle.bf16_to_f64(V[0][0, 0]) + oracle.bf16_to_f64(V[1][0, 0])) / 2,
                           rtol=1e-15, atol=1e-15)


# ---------------------------------------------------------------- invariants
def test_kv_slice_order_changes_only_rounding():
    rng = np.random.default_rng(2)
    P, H, S, d = 4, 2, 24, 32
    Q = [rand_bits((H, S, d), rng) for _ in range(P)]
    K = [rand_bits((H, S, d), rng) for _ in range(P)]
    V = [rand_bits((H, S, d), rng) for _ in range(P)]
    O, L, _ = full(Q, K, V)
    for perm in ([1, 2, 3, 0], [3, 2, 1, 0], [2, 0, 3, 1]):     # a ring started at another rank, ...
        O2, L2, _ = full(Q, [K[p] for p in perm], [V[p] for p in perm])
        assert np.abs(O2 - O).max() <= 1e-13 * np.abs(O).max()
        assert np.abs(L2 - L).max() <= 1e-13 * np.abs(L).max()


def test_a_common_key_offset_leaves_the_output_unchanged():
    rng = np.random.default_rng(3)
    P, H, S, d = 2, 1, 16, 8
    Q = [bits(rng.integers(-2, 3, (H, S, d)).astype(np.float64)) for _ in range(P)]
    Kv = [rng.integers(-2, 3, (H, S, d)).astype(np.float64) for _ in range(P)]
    V = [rand_bits((H, S, d), rng) for _ in range(P)]
    u = rng.integers(-3, 4, d).astype(np.float64)
    O, L, _ = full(Q, [bits(k) for k in Kv], V)
    O2, L2, _ = full(Q, [bits(k + u) for k in Kv], V)
    assert np.abs(O2 - O).max() <= 1e-13 * np.abs(O).max()
    for r in range(P):
        shift = oracle.bf16_to_f64(Q[r])[0] @ u / np.sqrt(d)   # every score of a query moves by q.u * scale
        assert np.allclose(L2[r, 0], L[r, 0] + shift, rtol=0, atol=1e-12)


def test_values_of_ones_give_ones():
    rng = np.random.default_rng(4)
    P, H, S, d = 3, 2, 20, 16
    Q = [rand_bits((H, S, d), rng, 2.0) for _ in range(P)]
    K = [rand_bits((H, S, d), rng, 2.0) for _ in range(P)]
    V = [bits(np.ones((H, S, d))) for _ in range(P)]
    O, _, _ = full(Q, K, V)
    assert np.abs(O - 1.0).max() <= 1e-15


# ---------------------------------------------------------------- library routine and brute force
@pytest.mark.parametrize("P,H,S,d", [(1, 1, 8, 16), (3, 2, 40, 32), (2, 3, 17, 128)])
def test_matches_numpy_softmax_attention(P, H, S, d):
    rng = np.random.default_rng(P * 100 + S)
    Q = [rand_bits((H, S, d), rng) for _ in range(P)]
    K = [rand_bits((H, S, d), rng) for _ in range(P)]
    V = [rand_bits((H, S, d), rng) for _ in range(P)]
    O, L, _ = full(Q, K, V)
    On, Ln = numpy_attention(Q, K, V)
    assert np.abs(O - On).max() <= 1e-13 * np.abs(On).max()
    assert np.abs(L - Ln).max() <= 1e-13 * np.abs(Ln).max()


def test_ring_attention_equals_its_rows():
    wl = ig.ATTN_WORKLOADS["ring_p2_h2_s256_d128"]
    Q, K, V = ig.make_attn_operands(wl)
    O, L, E = oracle.ring_attention(Q, K, V)
    rows = np.array([0, 5, 127, 128, 255])
    o, l, e = oracle.attention_rows(Q, K, V, 1, 1, rows)
    assert np.array_equal(O[1][1][rows], o) and np.array_equal(L[1][1][rows], l) and np.array_equal(E[1][1][rows], e)


@pytest.mark.parametrize("seed", [5, 6])
def test_bruteforce_50_digits(seed):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(seed)
    P, H, S, d = 2, 1, 3, 4
    Q = [rand_bits((H, S, d), rng, 1.5) for _ in range(P)]
    K = [rand_bits((H, S, d), rng, 1.5) for _ in range(P)]
    V = [rand_bits((H, S, d), rng) for _ in range(P)]
    O, L, E = full(Q, K, V)
    f = lambda x: [mpmath.mpf(float(v)) for v in oracle.bf16_to_f64(x).reshape(-1)]
    Kc = [f(K[o][0, j]) for o in range(P) for j in range(S)]
    Vc = [f(V[o][0, j]) for o in range(P) for j in range(S)]
    scale = 1 / mpmath.sqrt(d)
    for r in range(P):
        for i in range(S):
            q = f(Q[r][0, i])
            s = [scale * mpmath.fsum(a * b for a, b in zip(q, k)) for k in Kc]
            w = [mpmath.e ** x for x in s]
            l = mpmath.fsum(w)
            for c in range(d):
                want = mpmath.fsum(wj * v[c] for wj, v in zip(w, Vc)) / l
                assert abs(O[r, 0, i, c] - float(want)) <= 1e-14 * max(1.0, abs(float(want)))
                e = mpmath.sqrt(mpmath.fsum((wj * v[c]) ** 2 for wj, v in zip(w, Vc))) / l
                assert abs(E[r, 0, i, c] - float(e)) <= 1e-14 * float(e)
            assert abs(L[r, 0, i] - float(mpmath.log(l))) <= 1e-14 * max(1.0, abs(float(mpmath.log(l))))


# ---------------------------------------------------------------- planted mistakes trip a pin
MUTANTS = {
    "drops_last_rank": ("for (int o = 0; o < P; ++o)", "for (int o = 0; o < P - 1; ++o)"),
    "drops_last_key_row": ("for (int64_t j = 0; j < S; ++j)", "for (int64_t j = 0; j + 1 < S; ++j)"),
    "no_scale": ("const double sc = scale * dot;", "const double sc = dot;"),
    "scores_use_values": ("const uint16_t *krow = K[o] + (head * S + j) * d;",
                          "const uint16_t *krow = V[o] + (head * S + j) * d;"),
    "keys_of_head_0": ("const uint16_t *krow = K[o] + (head * S + j) * d;",
                       "const uint16_t *krow = K[o] + j * d;"),
    "queries_of_rank_0": ("const uint16_t *qrow = Q[rank] + (head * S + rows[t]) * d;",
                          "const uint16_t *qrow = Q[0] + (head * S + rows[t]) * d;"),
    "lse_without_max": ("lse[t] = m + log(l);", "lse[t] = log(l);"),
    "unnormalised": ("O[t * d + c] = acc[c] / l;", "O[t * d + c] = acc[c];"),
}


def _rows_fn(lib):
    def rows_fn(Q, K, V, rank, head, rows, scale=None):
        P = len(Q)
        H, S, d = Q[0].shape
        scale = 1 / np.sqrt(d) if scale is None else scale
        rows = np.ascontiguousarray(rows, np.int64)
        n = rows.size
        O = np.empty((n, d))
        E = np.empty((n, d))
        L = np.empty(n)
        arr = lambda xs: (ctypes.c_void_p * P)(*[x.ctypes.data for x in xs])
        lib.mko_attention_rows(P, ctypes.c_int64(H), ctypes.c_int64(S), ctypes.c_int64(d), arr(Q), arr(K), arr(V),
                               rank, ctypes.c_int64(head), ctypes.c_int64(n), rows.ctypes.data_as(ctypes.c_void_p),
                               ctypes.c_double(scale), O.ctypes.data_as(ctypes.c_void_p),
                               L.ctypes.data_as(ctypes.c_void_p), E.ctypes.data_as(ctypes.c_void_p))
        return O, L, E
    return rows_fn


def _pins_pass(lib):
    """The numpy comparison (H = 2, P = 3) and the one-dominant-key lse against a build."""
    rows_fn = _rows_fn(lib)
    rng = np.random.default_rng(7)
    P, H, S, d = 3, 2, 12, 16
    Q = [rand_bits((H, S, d), rng) for _ in range(P)]
    K = [rand_bits((H, S, d), rng) for _ in range(P)]
    V = [rand_bits((H, S, d), rng) for _ in range(P)]
    O, L, _ = full(Q, K, V, rows_fn)
    On, Ln = numpy_attention(Q, K, V)
    ok = np.abs(O - On).max() <= 1e-13 * np.abs(On).max() and np.abs(L - Ln).max() <= 1e-13 * np.abs(Ln).max()
    Qd = np.zeros((1, 1, 16))
    Qd[0, 0, 3] = 2048.0
    Kd = np.zeros((1, 1, 16))
    Kd[0, 0, 3] = 1.0
    O1, L1, _ = full([bits(Qd), bits(np.zeros((1, 1, 16)))], [bits(Kd), bits(np.zeros((1, 1, 16)))],
                     [bits(np.full((1, 1, 16), 2.0)), bits(np.full((1, 1, 16), -2.0))], rows_fn)
    return ok and L1[0, 0, 0] == 512.0 and np.all(O1[0, 0, 0] == 2.0)


def _build_variant(tmp_path, name, src):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                           str(so), str(c), "-lm"])
    lib = ctypes.CDLL(str(so))
    lib.mko_attention_rows.restype = None
    return lib


def test_planted_mistakes_are_caught(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mk_oracle_attn.c")).read()
    assert _pins_pass(_build_variant(tmp_path, "unmutated", src))
    for name, (old, new) in MUTANTS.items():
        assert old in src, name
        assert not _pins_pass(_build_variant(tmp_path, name, src.replace(old, new))), name
