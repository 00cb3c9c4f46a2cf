"""Failure detection without a GPU fault: a compute unit that is never produced (host-side
injection through mk_opts.debug_skip_unit) makes the consumer's bounded wait run out; the
kernel records MK_ERR_TIMEOUT, exits cleanly, and the next call on the same workspace and
context succeeds.  Also the controller trace and the device-side argument checks."""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gemm_tile_level_gb300 import api, mk
    import gpu_util as gu


@pytest.mark.parametrize("tiles", ["pair", "single"])
@pytest.mark.parametrize("split", ["adaptive", "static"])
def test_missing_unit_times_out_then_recovers(split, tiles):
    wl = ig.Workload("fault", "allreduce", 4, 512, 512, 128, ig.INTEGER_PM2, ig.INTEGER_PM2, "f32")
    A, B, Ad, Bd = gu.upload(wl)
    ws = api.workspace(mk.MK_OP_ALLREDUCE, 4, 512, 512, 128)
    mode = mk.MK_SPLIT_ADAPTIVE if split == "adaptive" else mk.MK_SPLIT_STATIC
    fl = mk.MK_FLAG_SINGLE_SM_TILES if tiles == "single" else 0
    o = api.make_opts(mode, comm_sms=4 if split == "static" else 0, timeout_ns=20_000_000, skip_unit=5, flags=fl)
    C, st = api.gemm_allreduce(Ad, Bd, mk.MK_F32, ws=ws, opts=o)
    assert st == mk.MK_OK                       # the launch itself is fine
    assert mk.mk_status_check(ws) == mk.MK_ERR_TIMEOUT
    assert "timed out" in mk.mk_last_error()
    assert mk.mk_status_check(ws) == mk.MK_OK   # read-and-clear
    C = gu.call_ar(Ad, Bd, mk.MK_F32, ws=ws,
                   opts=api.make_opts(mode, comm_sms=4 if split == "static" else 0, flags=fl))
    gu.assert_bit_exact(gu.host_values(C), oracle.allreduce(A, B))


@pytest.mark.parametrize("M,first_target", [(4096, 0), (256, 16)])
def test_controller_trace_records(M, first_target):
    """The controller's records: time, units and reduced tiles never go backwards; the target
    starts where the host put it (no reduce role in rank-major order, eight SM pairs in tile-major
    order) and is the whole grid once every compute unit has been claimed."""
    wl = ig.sweep_workload(M)
    A, B, Ad, Bd = gu.upload(wl)
    trace = torch.zeros(4096 * 32, dtype=torch.uint8, device="cuda")
    gu.call_ar(Ad, Bd, mk.MK_BF16, opts=api.make_opts(mk.MK_SPLIT_ADAPTIVE, trace=trace))
    rec = trace.cpu().numpy().view(np.dtype([("t", "<u8"), ("target", "<u4"), ("units", "<u4"),
                                             ("tiles", "<u4"), ("blocks", "<u4"), ("r", "<u8")]))
    n = int((rec["blocks"] > 0).sum())
    assert n > 2
    rec = rec[:n]
    S = gu.num_sms()
    assert (rec["blocks"] == S).all()
    assert (rec["target"] >= 0).all() and (rec["target"] <= S).all()
    assert rec["target"][0] == first_target
    assert rec["target"][-1] == S
    assert (np.diff(rec["t"].astype(np.int64)) >= 0).all()
    assert (np.diff(rec["units"].astype(np.int64)) >= 0).all()
    assert (np.diff(rec["tiles"].astype(np.int64)) >= 0).all()


def test_device_dependent_argument_checks():
    Ad = [torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Bd = [torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    S = gu.num_sms()
    _, st = api.gemm_allreduce(Ad, Bd, mk.MK_F32, opts=api.make_opts(mk.MK_SPLIT_STATIC, comm_sms=S))
    assert st == mk.MK_ERR_INVALID_ARG
    _, st = api.gemm_allreduce(Ad, Bd, mk.MK_F32, opts=api.make_opts(num_ctas=S + 1))
    assert st == mk.MK_ERR_NOT_RESIDENT
    _, st = api.gemm_allreduce(Ad, Bd, mk.MK_F32, opts=api.make_opts(num_ctas=7))
    assert st == mk.MK_ERR_INVALID_ARG      # SM pairs need an even grid
    # a smaller persistent grid is fine
    C = gu.call_ar(Ad, Bd, mk.MK_F32, opts=api.make_opts(num_ctas=8))
    assert not C.any()
