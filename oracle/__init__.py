"""fp64 CPU oracle for the rank-summed GEMM (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline / reference leg may
import this package.  It shares no code with the CUDA path (``gemm_tile_level_gb300``) and
does not import it.  The arithmetic lives in ``mk_oracle.c``; this file marshals numpy arrays.

Definitions followed (mKernel: Fast Multi-GPU, Multi-Node Fused Kernels, Table 3, the three
tensor-parallel rows):
  * GEMM + AllReduce:     every rank receives C = sum_r A_r B_r.
  * GEMM + ReduceScatter: rank s receives rows [s M/P, (s+1) M/P) of that same C.
  * AllGather + GEMM:     rank r receives [A_0; ...; A_{P-1}] B_r (row shards of A gathered,
                          B column-sharded).
Partial tiles stored at half width (bf16) are a variant of the boundary without a counterpart on
those pages: ``allreduce_bf16_partials`` defines it.
Ring Attention (the same Table 3, row "Ring Attention (SP)"; the arithmetic is in
``mk_oracle_attn.c``): every rank's queries attend, with softmax attention, to the keys and values
of the whole sequence, whose P slices the ring brings to each rank in turn.
Parity pins: every function here is pinned by tests/test_oracle_pins.py (the GEMM forms) and
tests/test_oracle_attention_pins.py (Ring Attention) against exact arithmetic, closed forms,
invariants, numpy's fp64 routines or a 50-digit brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mk_oracle.c")
_SRC_ATTN = os.path.join(_HERE, "mk_oracle_attn.c")
_LIB = os.path.join(_HERE, "_libmk_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2, OpenMP over rows, no FP contraction)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_ATTN))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
                               "-shared", "-o", tmp, _SRC, _SRC_ATTN, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.mko_gemm_rows.argtypes = [i64, i64, vp, vp, i64, i64, vp]
        lib.mko_rank_sum_rows.argtypes = [ctypes.c_int, i64, i64, vp, vp, i64, i64, vp]
        lib.mko_rank_sum_at.argtypes = [ctypes.c_int, i64, i64, vp, vp, i64, vp, vp, vp]
        lib.mko_round_bf16.argtypes = [vp, i64, vp]
        lib.mko_round_f32.argtypes = [vp, i64, vp]
        lib.mko_attention_rows.argtypes = [ctypes.c_int, i64, i64, i64, vp, vp, vp, ctypes.c_int, i64, i64, vp,
                                           ctypes.c_double, vp, vp, vp]
        for f in (lib.mko_gemm_rows, lib.mko_rank_sum_rows, lib.mko_rank_sum_at,
                  lib.mko_round_bf16, lib.mko_round_f32, lib.mko_attention_rows):
            f.restype = None
        _lib = lib
    return _lib


def _bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return x


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _check_ranks(A, B):
    P = len(A)
    if P == 0 or len(B) != P:
        raise ValueError("need P >= 1 matching A_r, B_r")
    M, Kr = A[0].shape
    N = B[0].shape[1]
    for a, b in zip(A, B):
        if a.shape != (M, Kr) or b.shape != (Kr, N):
            raise ValueError("inconsistent rank shapes")
    return P, M, N, Kr


def gemm(X, Y) -> np.ndarray:
    """Plain fp64 product X @ Y of two bf16-bit matrices."""
    X, Y = _bits(X), _bits(Y)
    m, k = X.shape
    k2, n = Y.shape
    assert k == k2
    out = np.empty((m, n), np.float64)
    if m and n:
        _load().mko_gemm_rows(n, k, X.ctypes.data, Y.ctypes.data, 0, m, out.ctypes.data)
    return out


def allreduce_rows(A, B, i0: int, ni: int) -> np.ndarray:
    """Rows [i0, i0+ni) of C = sum_r A_r B_r in fp64 (rank order 0..P-1)."""
    A = [_bits(a) for a in A]
    B = [_bits(b) for b in B]
    P, M, N, Kr = _check_ranks(A, B)
    assert 0 <= i0 and i0 + ni <= M
    out = np.empty((ni, N), np.float64)
    if ni and N:
        _load().mko_rank_sum_rows(P, N, Kr, _ptr_array(A), _ptr_array(B), i0, ni, out.ctypes.data)
    return out


def allreduce(A, B) -> np.ndarray:
    """GEMM + AllReduce: the full C = sum_r A_r B_r (M x N, fp64)."""
    return allreduce_rows(A, B, 0, A[0].shape[0])


def allreduce_at(A, B, rows, cols) -> np.ndarray:
    """C[rows[s], cols[s]] for each sample s, same operation order as ``allreduce``."""
    A = [_bits(a) for a in A]
    B = [_bits(b) for b in B]
    P, M, N, Kr = _check_ranks(A, B)
    rows = np.ascontiguousarray(rows, np.int64)
    cols = np.ascontiguousarray(cols, np.int64)
    assert rows.shape == cols.shape
    assert (rows >= 0).all() and (rows < M).all() and (cols >= 0).all() and (cols < N).all()
    out = np.empty(rows.shape, np.float64)
    if rows.size:
        _load().mko_rank_sum_at(P, N, Kr, _ptr_array(A), _ptr_array(B), rows.size,
                                rows.ctypes.data, cols.ctypes.data, out.ctypes.data)
    return out


def allreduce_bf16_partials(A, B) -> np.ndarray:
    """The bf16-partial-tile form of GEMM + AllReduce: sum_r RNE_bf16(A_r B_r), summed in fp64 in
    rank order.  Each per-rank partial product is rounded to bf16 (round to nearest even) before
    the ranks are added, which is what storing partial tiles at half width computes.  The partial
    is rounded from its fp64 value here; a kernel that rounds its fp32 accumulator lands on the
    other side of a rounding midpoint only where the two differ across it.
    Parity pinned (ties-to-even closed form, reduction to ``allreduce`` when every partial is
    exact in bf16, exact-rational brute force)."""
    A = [_bits(a) for a in A]
    B = [_bits(b) for b in B]
    P, M, N, Kr = _check_ranks(A, B)
    out = np.zeros((M, N), np.float64)
    for a, b in zip(A, B):
        out += bf16_to_f64(round_bf16(gemm(a, b)))
    return out


def allreduce_bf16_partials_at(A, B, rows, cols) -> np.ndarray:
    """``allreduce_bf16_partials`` at the sampled elements (rows[s], cols[s]) only."""
    out = np.zeros(np.asarray(rows).shape, np.float64)
    for a, b in zip(A, B):
        out += bf16_to_f64(round_bf16(allreduce_at([a], [b], rows, cols)))
    return out


def reducescatter(A, B):
    """GEMM + ReduceScatter: shard s is rows [s M/P, (s+1) M/P) of sum_r A_r B_r."""
    P, M, N, Kr = _check_ranks(A, B)
    if M % P:
        raise ValueError("M must be divisible by P")
    C = allreduce(A, B)
    h = M // P
    return [C[s * h:(s + 1) * h] for s in range(P)]


def allgather_gemm(A_shards, B_cols):
    """AllGather + GEMM: C_r = [A_0; ...; A_{P-1}] @ B_r for every rank r."""
    A_cat = np.concatenate([_bits(a) for a in A_shards], axis=0)
    return [gemm(A_cat, b) for b in B_cols]


def round_bf16(x) -> np.ndarray:
    """fp64 -> bf16 bits, round to nearest even applied to the fp64 value."""
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    if x.size:
        _load().mko_round_bf16(x.ctypes.data, x.size, out.ctypes.data)
    return out


def round_f32(x) -> np.ndarray:
    """fp64 -> fp32, round to nearest even."""
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, np.float32)
    if x.size:
        _load().mko_round_f32(x.ctypes.data, x.size, out.ctypes.data)
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64 (for comparisons)."""
    bits = np.asarray(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- Ring Attention
def _check_attn(Q, K, V):
    P = len(Q)
    if P == 0 or len(K) != P or len(V) != P:
        raise ValueError("need P >= 1 matching Q_r, K_r, V_r")
    H, S, d = Q[0].shape
    for x in list(Q) + list(K) + list(V):
        if x.shape != (H, S, d):
            raise ValueError("inconsistent rank shapes (each rank holds H x S x d)")
    return P, H, S, d


def attention_rows(Q, K, V, rank: int, head: int, rows, scale: float | None = None):
    """Softmax attention of query rows ``rows`` of head ``head`` on rank ``rank`` over the keys and
    values of every rank (fp64).  Q, K, V: lists of P arrays of bf16 bits, each H x S x d.  Returns
    (O [n x d], lse [n], err [n x d]); lse is the natural-log logsumexp of the scaled scores and
    err the scale of the error that rounding each probability would add (see mk_oracle_attn.c).
    ``scale`` defaults to 1/sqrt(d)."""
    Q = [_bits(x) for x in Q]
    K = [_bits(x) for x in K]
    V = [_bits(x) for x in V]
    P, H, S, d = _check_attn(Q, K, V)
    rows = np.ascontiguousarray(rows, np.int64)
    assert 0 <= rank < P and 0 <= head < H and ((rows >= 0) & (rows < S)).all()
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    n = rows.size
    O = np.empty((n, d), np.float64)
    err = np.empty((n, d), np.float64)
    lse = np.empty(n, np.float64)
    if n and d:
        _load().mko_attention_rows(P, H, S, d, _ptr_array(Q), _ptr_array(K), _ptr_array(V), rank, head, n,
                                   rows.ctypes.data, float(scale), O.ctypes.data, lse.ctypes.data, err.ctypes.data)
    return O, lse, err


def ring_attention(Q, K, V, scale: float | None = None):
    """The whole Ring Attention result: per rank, O_r (H x S x d), lse_r (H x S) and err_r (H x S x d),
    fp64."""
    P, H, S, d = _check_attn(Q, K, V)
    outs, lses, errs = [], [], []
    rows = np.arange(S, dtype=np.int64)
    for r in range(P):
        O = np.empty((H, S, d))
        L = np.empty((H, S))
        E = np.empty((H, S, d))
        for h in range(H):
            O[h], L[h], E[h] = attention_rows(Q, K, V, r, h, rows, scale)
        outs.append(O)
        lses.append(L)
        errs.append(E)
    return outs, lses, errs
