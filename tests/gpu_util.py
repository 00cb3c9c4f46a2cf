"""Shared helpers of the GPU tests: upload seeded inputs, run the C ABI, compare to the oracle.

Tolerances (the reading of the stated bounds, applied per output dtype):
  fp32 output : max|err| <= 1e-2 * rms(C_ref)  and  ||err||_F / ||C_ref||_F <= 2e-3
  bf16 output : ||err||_F / ||C_ref||_F <= 2e-3  and, elementwise,
                |err| <= 1e-2 * rms(C_ref) + ulp_bf16(C_ref)
                (a correctly rounded bf16 result already misses the bare 1e-2*rms bound in the
                tails, where half an ulp exceeds it)
  integer-valued inputs : bit-exact (every partial sum is an integer below 2^24, so fp32
                accumulation is exact in any order and both sides round the same integer).
"""
from __future__ import annotations

import numpy as np
import torch

import inputgen as ig
import oracle
from gemm_tile_level_gb300 import api, mk


def upload(wl: ig.Workload, integer=False):
    w = wl.integer_variant() if integer else wl
    A, B = ig.make_operands(w)
    return A, B, [api.bf16_device(a) for a in A], [api.bf16_device(b) for b in B]


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host_values(t: torch.Tensor) -> np.ndarray:
    """Result tensor -> fp64 numpy (bf16 widened exactly)."""
    if t.dtype == torch.bfloat16:
        return oracle.bf16_to_f64(host_bits(t))
    return t.cpu().numpy().astype(np.float64)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126)
    return np.exp2(e - 7)


def check_tolerance(out: np.ndarray, ref: np.ndarray, out_bf16: bool, rms_ref: float | None = None):
    """Assert the stated tolerances; rms_ref may come from the full reference when `ref` is a
    sample of it."""
    err = out - ref
    rms = float(np.sqrt(np.mean(ref ** 2))) if rms_ref is None else rms_ref
    rel_f = float(np.linalg.norm(err) / np.linalg.norm(ref))
    assert rel_f <= 2e-3, f"relative Frobenius error {rel_f:.3e}"
    if out_bf16:
        bad = np.abs(err) > 1e-2 * rms + ulp_bf16(ref)
    else:
        bad = np.abs(err) > 1e-2 * rms
    assert not bad.any(), f"{int(bad.sum())} elements beyond bound; worst {np.abs(err).max():.3e} (rms {rms:.3e})"
    return rel_f, float(np.abs(err).max() / rms)


def assert_bit_exact(out: np.ndarray, ref_rounded: np.ndarray):
    """Exact equality of values (IEEE equality: +0 == -0)."""
    mism = out != ref_rounded
    assert not mism.any(), f"{int(mism.sum())} mismatches, first at {np.argwhere(mism)[0]}"


def rounded_reference(ref: np.ndarray, out_bf16: bool) -> np.ndarray:
    if out_bf16:
        return oracle.bf16_to_f64(oracle.round_bf16(ref))
    return oracle.round_f32(ref).astype(np.float64)


def sample_indices(M, N, n=4096, seed=0):
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n))
    cols = list(rng.integers(0, N, n))
    for r in (0, min(127, M - 1), min(128, M - 1), M - 1):
        for c in (0, min(127, N - 1), min(128, N - 1), min(255, N - 1), min(256, N - 1), N - 1):
            rows.append(r)
            cols.append(c)
    return np.array(rows, np.int64), np.array(cols, np.int64)


def call_ar(Ad, Bd, out_dtype, opts=None, ws=None, C=None):
    """mk_gemm_allreduce + status check; returns the result tensor (or list)."""
    P = len(Ad)
    M, Kr = Ad[0].shape
    N = Bd[0].shape[1]
    if ws is None:
        ws = api.workspace(mk.MK_OP_ALLREDUCE, P, M, N, Kr)
    C, st = api.gemm_allreduce(Ad, Bd, out_dtype, C=C, ws=ws, opts=opts)
    mk.check(st)
    mk.check(mk.mk_status_check(ws))
    return C


def call_rs(Ad, Bd, out_dtype, opts=None, ws=None):
    P = len(Ad)
    M, Kr = Ad[0].shape
    N = Bd[0].shape[1]
    if ws is None:
        ws = api.workspace(mk.MK_OP_REDUCESCATTER, P, M, N, Kr)
    shards, st = api.gemm_reducescatter(Ad, Bd, out_dtype, ws=ws, opts=opts)
    mk.check(st)
    mk.check(mk.mk_status_check(ws))
    return shards


def num_sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count
