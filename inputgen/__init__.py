"""Seeded synthetic inputs for the rank-summed GEMM workloads.

This module is shared by the tests, the bench and the oracle's callers.  It only
draws bf16 bit patterns (Philox4x32-10 counter streams, see ``philox_gen.c``) and
describes the workload shapes; it does none of the GEMM or reduction arithmetic.

Operand layout (row-parallel tensor parallelism, K split across P logical ranks):
  A_r : M x K_r   bf16, row-major (K contiguous)
  B_r : K_r x N   bf16, row-major (N contiguous)
Stream of tensor ``tid`` of rank ``r``: Philox key (seed, r), counter
(element block, tid); A uses tid 0 and B uses tid 1.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "philox_gen.c")
_LIB = os.path.join(_HERE, "_libinputgen.so")

DIST_UNIFORM, DIST_NORMAL, DIST_INTEGER = 0, 1, 2
TID_A, TID_B = 0, 1

_lib = None


def build(force: bool = False) -> str:
    """Compile the generator into ``_libinputgen.so`` (gcc, OpenMP, no FP contraction
    so x86 and Arm hosts draw identical values)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.ig_philox4x32_10.argtypes = [ctypes.POINTER(ctypes.c_uint32)] * 3
        lib.ig_philox4x32_10.restype = None
        lib.ig_fill_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_double, ctypes.c_double, ctypes.c_uint32,
                                     ctypes.c_uint32, ctypes.c_uint32]
        lib.ig_fill_bf16.restype = ctypes.c_int
        _lib = lib
    return _lib


def philox4x32_10(ctr, key):
    """One Philox4x32-10 block: four 32-bit words for counter ``ctr`` (4 words), key ``key`` (2 words)."""
    lib = _load()
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (ctypes.c_uint32 * 4)()
    lib.ig_philox4x32_10(c, k, o)
    return tuple(int(x) for x in o)


def fill_bf16(out: np.ndarray, dist, seed: int, rank: int, tid: int, first: int = 0) -> np.ndarray:
    """Fill the contiguous uint16 array ``out`` with elements [first, first+out.size) of the
    stream (seed, rank, tid) drawn from ``dist`` = (kind, p0, p1)."""
    assert out.dtype == np.uint16 and out.flags["C_CONTIGUOUS"]
    kind, p0, p1 = dist
    rc = _load().ig_fill_bf16(out.ctypes.data, int(first), int(out.size), int(kind), float(p0),
                              float(p1), int(seed) & 0xFFFFFFFF, int(rank), int(tid))
    if rc != 0:
        raise ValueError(f"unknown distribution {dist}")
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """View bf16 bit patterns as float32 values (exact widening)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


UNIFORM_PM1 = (DIST_UNIFORM, -1.0, 1.0)
INTEGER_PM2 = (DIST_INTEGER, -2.0, 2.0)


def normal(var: float):
    """N(0, var): the second parameter is the variance."""
    return (DIST_NORMAL, 0.0, float(var))


@dataclass(frozen=True)
class Workload:
    """One seeded synthetic problem: C = sum_r A_r B_r over P logical ranks."""
    name: str
    op: str                     # "allreduce" or "reducescatter"
    P: int
    M: int
    N: int
    Kr: int
    a_dist: tuple
    b_dist: tuple
    out_dtype: str              # "f32" or "bf16"
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.Kr * self.P

    def integer_variant(self) -> "Workload":
        return Workload(self.name + "_int", self.op, self.P, self.M, self.N, self.Kr, INTEGER_PM2,
                        INTEGER_PM2, self.out_dtype, self.seed, "entries in {-2..2}")

    def with_shape(self, **kw) -> "Workload":
        d = dict(name=self.name, op=self.op, P=self.P, M=self.M, N=self.N, Kr=self.Kr,
                 a_dist=self.a_dist, b_dist=self.b_dist, out_dtype=self.out_dtype, seed=self.seed)
        d.update(kw)
        return Workload(**d)


def make_operands(wl: Workload, out_a=None, out_b=None):
    """Return ([A_0..A_{P-1}], [B_0..B_{P-1}]) as uint16 bf16-bit arrays (or fill the given
    contiguous arrays in place)."""
    A, B = [], []
    for r in range(wl.P):
        a = out_a[r] if out_a is not None else np.empty((wl.M, wl.Kr), np.uint16)
        b = out_b[r] if out_b is not None else np.empty((wl.Kr, wl.N), np.uint16)
        fill_bf16(a.reshape(-1), wl.a_dist, wl.seed, r, TID_A)
        fill_bf16(b.reshape(-1), wl.b_dist, wl.seed, r, TID_B)
        A.append(a)
        B.append(b)
    return A, B


# The five workloads of the method's tensor-parallel GEMM+collective study, sized for one GPU.
WORKLOADS = {
    "ar_p2_m128_n128_k256": Workload("ar_p2_m128_n128_k256", "allreduce", 2, 128, 128, 256,
                                     UNIFORM_PM1, normal(1 / 512), "f32"),
    "ar_p8_m2048_n4096_k512": Workload("ar_p8_m2048_n4096_k512", "allreduce", 8, 2048, 4096, 512,
                                       UNIFORM_PM1, normal(1 / 4096), "bf16"),
    "ar_mlp_down_p8_m8192_n8192_k3584": Workload("ar_mlp_down_p8_m8192_n8192_k3584", "allreduce", 8,
                                                 8192, 8192, 3584, normal(1.0), normal(1 / 28672),
                                                 "bf16"),
    "rs_p8_m16384_n8192_k1024": Workload("rs_p8_m16384_n8192_k1024", "reducescatter", 8, 16384, 8192,
                                         1024, UNIFORM_PM1, normal(1 / 8192), "bf16"),
}
SWEEP_M = (256, 512, 1024, 2048, 4096, 8192, 16384)


def sweep_workload(M: int) -> Workload:
    """The SM-split sweep: GEMM+AllReduce, P=8, N=8192, K_r=1024, A ~ N(0,1), B ~ N(0,1/8192)."""
    return Workload(f"ar_sweep_p8_m{M}_n8192_k1024", "allreduce", 8, M, 8192, 1024, normal(1.0),
                    normal(1 / 8192), "bf16")


# ---------------------------------------------------------------- Ring Attention (sequence parallel)
TID_Q, TID_K, TID_V = 2, 3, 4


@dataclass(frozen=True)
class AttnWorkload:
    """One seeded Ring Attention problem: P ranks, each holding a slice of S tokens of the sequence
    as Q_r, K_r, V_r (H heads x S rows x d, bf16, row-major)."""
    name: str
    P: int
    H: int
    S: int
    d: int
    q_dist: tuple
    k_dist: tuple
    v_dist: tuple
    out_dtype: str = "bf16"
    seed: int = 0

    @property
    def flops(self) -> int:
        """Q K^T and P V over the whole sequence: 4 * (P S)^2 * d per head."""
        return 4 * (self.P * self.S) ** 2 * self.d * self.H

    def with_shape(self, **kw) -> "AttnWorkload":
        d = dict(name=self.name, P=self.P, H=self.H, S=self.S, d=self.d, q_dist=self.q_dist,
                 k_dist=self.k_dist, v_dist=self.v_dist, out_dtype=self.out_dtype, seed=self.seed)
        d.update(kw)
        return AttnWorkload(**d)


def make_attn_operands(wl: AttnWorkload):
    """Return ([Q_r], [K_r], [V_r]) as uint16 bf16-bit arrays of shape (H, S, d), one per rank."""
    Q, K, V = [], [], []
    for r in range(wl.P):
        for lst, dist, tid in ((Q, wl.q_dist, TID_Q), (K, wl.k_dist, TID_K), (V, wl.v_dist, TID_V)):
            x = np.empty((wl.H, wl.S, wl.d), np.uint16)
            fill_bf16(x.reshape(-1), dist, wl.seed, r, tid)
            lst.append(x)
    return Q, K, V


# Sequence-parallel attention: a small case the oracle finishes in seconds, and a long-context
# case (8 ranks x 4096 tokens = 32768 tokens, 32 heads of 128) for the bench.
ATTN_WORKLOADS = {
    "ring_p2_h2_s256_d128": AttnWorkload("ring_p2_h2_s256_d128", 2, 2, 256, 128, normal(1.0), normal(1.0),
                                         normal(1.0)),
    "ring_p8_h32_s4096_d128": AttnWorkload("ring_p8_h32_s4096_d128", 8, 32, 4096, 128, normal(1.0), normal(1.0),
                                           normal(1.0)),
    # the same sequence with 8 heads: a case small enough for a full profiler capture
    "ring_p8_h8_s4096_d128": AttnWorkload("ring_p8_h8_s4096_d128", 8, 8, 4096, 128, normal(1.0), normal(1.0),
                                          normal(1.0)),
}
