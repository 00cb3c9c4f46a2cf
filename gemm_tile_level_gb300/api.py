"""torch-tensor helpers around the C ABI: allocate device buffers and the workspace, call.

torch supplies device memory and the stream; every step of the computation runs in libmk.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import mk

_TORCH_OUT = {mk.MK_BF16: torch.bfloat16, mk.MK_F32: torch.float32}


def bf16_device(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """Upload a uint16 array of bf16 bit patterns as a contiguous bf16 device tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16)
    return t.to(device)


def workspace(op: int, P: int, M: int, N: int, K_per_rank: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace of the size the op needs (torch allocations are 512-byte aligned)."""
    n = mk.mk_workspace_size(op, P, M, N, K_per_rank)
    if n == 0:
        raise ValueError("invalid shape for mk_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def make_opts(split_mode=mk.MK_SPLIT_ADAPTIVE, comm_sms=0, timeout_ns=0, trace=None, num_ctas=0,
              flags=0, skip_unit=-1, raster_group=0, reduce_split=0, chain_ranks=0) -> mk.mk_opts:
    o = mk.mk_opts_default()
    o.split_mode = split_mode
    o.comm_sms = comm_sms
    if timeout_ns:
        o.wait_timeout_ns = timeout_ns
    if trace is not None:
        o.trace = trace.data_ptr()
        o.trace_bytes = trace.numel() * trace.element_size()
    o.num_ctas = num_ctas
    o.flags = flags
    o.debug_skip_unit = skip_unit
    o.raster_group = raster_group
    o.reduce_split = reduce_split
    o.chain_ranks = chain_ranks
    return o


def gemm_allreduce(A, B, out_dtype=mk.MK_BF16, C=None, ws=None, opts=None, stream=None):
    """C = sum_r A[r] @ B[r] via mk_gemm_allreduce.  Returns (C, status).  C may be one tensor
    (every rank shares it) or a list of P tensors."""
    P = len(A)
    M, Kr = A[0].shape
    N = B[0].shape[1]
    if C is None:
        C = torch.empty((M, N), dtype=_TORCH_OUT[out_dtype], device=A[0].device)
    Cs = C if isinstance(C, (list, tuple)) else [C] * P
    if ws is None:
        ws = workspace(mk.MK_OP_ALLREDUCE, P, M, N, Kr, A[0].device)
    st = mk.mk_gemm_allreduce(P, M, N, Kr, A, B, Cs, out_dtype, ws, opts=opts, stream=stream)
    return C, st


def gemm_reducescatter(A, B, out_dtype=mk.MK_BF16, shards=None, ws=None, opts=None, stream=None):
    """Row shard s of sum_r A[r] @ B[r] into shards[s] via mk_gemm_reducescatter."""
    P = len(A)
    M, Kr = A[0].shape
    N = B[0].shape[1]
    if shards is None:
        shards = [torch.empty((M // P, N), dtype=_TORCH_OUT[out_dtype], device=A[0].device)
                  for _ in range(P)]
    if ws is None:
        ws = workspace(mk.MK_OP_REDUCESCATTER, P, M, N, Kr, A[0].device)
    st = mk.mk_gemm_reducescatter(P, M, N, Kr, A, B, shards, out_dtype, ws, opts=opts, stream=stream)
    return shards, st


def allgather_gemm(A_shards, B, out_dtype=mk.MK_BF16, gather=True, C=None, gathered=None, ws=None, opts=None,
                   stream=None):
    """C[r] = [A_shards[0]; ...; A_shards[P-1]] @ B[r] via mk_allgather_gemm.  With gather=True the
    shards are also copied into P gathered buffers (returned); otherwise they are read in place.
    Returns (C, gathered, status)."""
    P = len(A_shards)
    Mp, K = A_shards[0].shape
    M = Mp * P
    N = B[0].shape[1]
    dev = A_shards[0].device
    if C is None:
        C = [torch.empty((M, N), dtype=_TORCH_OUT[out_dtype], device=dev) for _ in range(P)]
    if gather and gathered is None:
        gathered = [torch.empty((M, K), dtype=torch.bfloat16, device=dev) for _ in range(P)]
    if ws is None:
        ws = workspace(mk.MK_OP_ALLGATHER_GEMM, P, M, N, K, dev)
    st = mk.mk_allgather_gemm(P, M, N, K, A_shards, B, gathered if gather else None, C, out_dtype, ws, opts=opts,
                              stream=stream)
    return C, gathered, st


def ring_attention_workspace(P: int, H: int, S: int, d: int, device="cuda") -> torch.Tensor:
    """A zeroed Ring Attention workspace (header and one flag per forwarded KV tile)."""
    n = mk.mk_ring_attention_workspace_size(P, H, S, d)
    if n == 0:
        raise ValueError("invalid shape for mk_ring_attention_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def ring_attention(Q, K, V, out_dtype=mk.MK_BF16, scale=0.0, ring=True, lse=True, O=None, kv_ring=None, ws=None,
                   opts=None, stream=None):
    """O[r] = softmax(scale Q[r] K_all^T) V_all via mk_ring_attention; Q[r], K[r], V[r] are H x S x d
    bf16 tensors.  With ring=True the KV slices are forwarded around the ring through P receive
    buffers (returned).  Returns (O, lse, kv_ring, status)."""
    P = len(Q)
    H, S, d = Q[0].shape
    dev = Q[0].device
    if O is None:
        O = [torch.empty((H, S, d), dtype=_TORCH_OUT[out_dtype], device=dev) for _ in range(P)]
    L = [torch.empty((H, S), dtype=torch.float32, device=dev) for _ in range(P)] if lse else None
    if ring and kv_ring is None and P > 1:
        kv_ring = [torch.empty((P - 1, 2, H, S, d), dtype=torch.bfloat16, device=dev) for _ in range(P)]
    if ws is None:
        ws = ring_attention_workspace(P, H, S, d, dev)
    st = mk.mk_ring_attention(P, H, S, d, Q, K, V, O, L, kv_ring if ring else None, out_dtype, scale, ws,
                              opts=opts, stream=stream)
    return O, L, kv_ring, st
