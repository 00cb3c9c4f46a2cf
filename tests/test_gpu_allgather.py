"""AllGather + GEMM (column-parallel tensor parallelism) through the C ABI against the oracle.

mKernel: Fast Multi-GPU, Multi-Node Fused Kernels, Table 3, row "AllGather + GEMM (TP)":
communication precedes compute; rank r receives [A_0; ...; A_{P-1}] B_r.  Communication-role
blocks copy 128-row chunks of the shards into every rank's gathered buffer and release a flag
per chunk; compute-role blocks acquire the flags of the rows they load.
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


def make(P, M, N, K, dist_a, dist_b, seed=1):
    A = [np.empty((M // P, K), np.uint16) for _ in range(P)]
    B = [np.empty((K, N), np.uint16) for _ in range(P)]
    for r in range(P):
        ig.fill_bf16(A[r].reshape(-1), dist_a, seed, r, ig.TID_A)
        ig.fill_bf16(B[r].reshape(-1), dist_b, seed, r, ig.TID_B)
    return A, B, [api.bf16_device(a) for a in A], [api.bf16_device(b) for b in B]


def run(Ad, Bd, code, gather=True, split="fused", comm_sms=0):
    mode = mk.MK_SPLIT_UNFUSED if split == "unfused" else mk.MK_SPLIT_ADAPTIVE
    P = len(Ad)
    Mp, K = Ad[0].shape
    ws = api.workspace(mk.MK_OP_ALLGATHER_GEMM, P, Mp * P, Bd[0].shape[1], K)
    C, G, st = api.allgather_gemm(Ad, Bd, code, gather=gather, ws=ws, opts=api.make_opts(mode, comm_sms=comm_sms))
    mk.check(st)
    mk.check(mk.mk_status_check(ws))
    return C, G


SHAPES = [
    # P, M, N, K
    (2, 256, 128, 256),
    (3, 192, 136, 72),      # 64-row shards (gathered path only), ragged N, K below one slice
    (4, 1024, 264, 200),
    (8, 2048, 512, 512),
    (1, 130, 8, 8),
    (16, 2048, 264, 136),   # the most ranks, ragged N and K
]


@pytest.mark.parametrize("P,M,N,K", SHAPES)
@pytest.mark.parametrize("split", ["fused", "unfused"])
def test_integer_bit_exact_and_gathered_copies(P, M, N, K, split):
    A, B, Ad, Bd = make(P, M, N, K, ig.INTEGER_PM2, ig.INTEGER_PM2, seed=P + M)
    want = oracle.allgather_gemm(A, B)
    C, G = run(Ad, Bd, mk.MK_F32, split=split)
    cat = np.concatenate(A, axis=0)
    for r in range(P):
        gu.assert_bit_exact(gu.host_values(C[r]), want[r])
        assert np.array_equal(gu.host_bits(G[r]), cat)


@pytest.mark.parametrize("P,M,N,K", [(2, 256, 128, 256), (4, 1024, 264, 200), (8, 2048, 512, 512)])
def test_shards_read_in_place(P, M, N, K):
    A, B, Ad, Bd = make(P, M, N, K, ig.INTEGER_PM2, ig.INTEGER_PM2, seed=5)
    want = oracle.allgather_gemm(A, B)
    C, _ = run(Ad, Bd, mk.MK_BF16, gather=False)
    for r in range(P):
        gu.assert_bit_exact(gu.host_values(C[r]), gu.rounded_reference(want[r], True))


def test_random_within_tolerance_and_split_invariant():
    P, M, N, K = 8, 4096, 1024, 2048
    A, B, Ad, Bd = make(P, M, N, K, ig.normal(1.0), ig.normal(1.0 / K), seed=9)
    rows, cols = gu.sample_indices(M, N, 1024)
    Acat = np.concatenate(A, axis=0)
    C, _ = run(Ad, Bd, mk.MK_BF16)
    C2, _ = run(Ad, Bd, mk.MK_BF16, split="unfused")
    C3, _ = run(Ad, Bd, mk.MK_BF16, comm_sms=40)
    for r in (0, P - 1):
        ref = oracle.allreduce_at([Acat], [B[r]], rows, cols)
        rms = float(np.sqrt(np.mean(oracle.allreduce_rows([Acat], [B[r]], 0, 2) ** 2)))
        gu.check_tolerance(gu.host_values(C[r])[rows, cols], ref, out_bf16=True, rms_ref=rms)
    for r in range(P):
        assert torch.equal(C[r], C2[r]) and torch.equal(C[r], C3[r])


def test_argument_checks():
    P, M, N, K = 4, 512, 128, 64
    _, _, Ad, Bd = make(P, M, N, K, ig.INTEGER_PM2, ig.INTEGER_PM2)
    ws = api.workspace(mk.MK_OP_ALLGATHER_GEMM, P, M, N, K)
    C = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    G = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    st = mk.mk_allgather_gemm(P, M, N, K, Ad, Bd, [G[0], None, G[2], G[3]], C, mk.MK_BF16, ws)
    assert st == mk.MK_ERR_INVALID_ARG
    st = mk.mk_allgather_gemm(3, 512, N, K, Ad[:3], Bd[:3], None, C[:3], mk.MK_BF16, ws)
    assert st == mk.MK_ERR_UNSUPPORTED_SHAPE          # M not divisible by P
    st = mk.mk_allgather_gemm(4, 256, N, K, Ad, Bd, None, C, mk.MK_BF16, ws)
    assert st == mk.MK_ERR_UNSUPPORTED_SHAPE          # 64-row shards need gathered buffers


@pytest.mark.parametrize("split", ["fused", "unfused"])
def test_benchmarked_shape_every_rank(split):
    """The column-parallel MLP up-projection the bench times: P=8, M=8192 tokens, K=4096, 3584
    output columns per rank.  Every rank is checked on sampled elements against the oracle, bit
    for bit on integer-valued inputs and within the tolerance on random ones; every gathered copy
    must equal the concatenated shards."""
    P, M, N, K = 8, 8192, 3584, 4096
    rows, cols = gu.sample_indices(M, N, 2048, seed=3)
    for integer in (True, False):
        if integer:
            A, B, Ad, Bd = make(P, M, N, K, ig.INTEGER_PM2, ig.INTEGER_PM2, seed=21)
        else:
            A, B, Ad, Bd = make(P, M, N, K, ig.normal(1.0), ig.normal(1.0 / K), seed=0)
        C, G = run(Ad, Bd, mk.MK_BF16, split=split)
        Acat = np.concatenate(A, axis=0)
        cat_dev = torch.cat(Ad, dim=0)
        for r in range(P):
            ref = oracle.allreduce_at([Acat], [B[r]], rows, cols)
            got = gu.host_values(C[r])[rows, cols]
            if integer:
                gu.assert_bit_exact(got, gu.rounded_reference(ref, True))
            else:
                rms = float(np.sqrt(np.mean(oracle.allreduce_rows([Acat], [B[r]], 0, 2) ** 2)))
                gu.check_tolerance(got, ref, out_bf16=True, rms_ref=rms)
            assert torch.equal(G[r], cat_dev), f"gathered copy of rank {r} differs from the shards"
        del C, G, Ad, Bd, cat_dev
        torch.cuda.empty_cache()


def test_benchmarked_shape_every_element():
    """The bench's AllGather + GEMM shape (P=8, M=8192, K=4096, 3584 columns per rank) on random
    inputs, fused: every element of every rank's output against the fp64 oracle (about 35 s of
    the oracle on the GPU host's cores)."""
    P, M, N, K = 8, 8192, 3584, 4096
    A, B, Ad, Bd = make(P, M, N, K, ig.normal(1.0), ig.normal(1.0 / K), seed=0)
    C, G = run(Ad, Bd, mk.MK_BF16)
    got = [gu.host_values(c) for c in C]
    del C, G, Ad, Bd
    torch.cuda.empty_cache()
    for r, ref in enumerate(oracle.allgather_gemm(A, B)):
        gu.check_tolerance(got[r], ref, out_bf16=True)
