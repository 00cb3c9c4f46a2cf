"""The C ABI on a machine without a GPU: the library loads, exports every symbol mk.h
declares, its structs match the binding, the workspace arithmetic, and the argument checks
that return before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mk.h")


@pytest.fixture(scope="module")
def mk():
    from gemm_tile_level_gb300 import build
    build.build()
    from gemm_tile_level_gb300 import mk as mkmod
    return mkmod


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(mk):
    names = declared_functions()
    assert set(names) == set(mk.EXPORTED)
    lib = ctypes.CDLL(mk.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", mk.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", out, re.M), n


def test_struct_layout_matches_header(mk, tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "mk.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(mk_opts), offsetof(mk_opts, comm_sms),
         offsetof(mk_opts, wait_timeout_ns), offsetof(mk_opts, trace), offsetof(mk_opts, trace_bytes),
         offsetof(mk_opts, num_ctas), offsetof(mk_opts, flags), offsetof(mk_opts, debug_skip_unit),
         sizeof(mk_trace_record), offsetof(mk_opts, raster_group), offsetof(mk_opts, reduce_split),
         offsetof(mk_opts, chain_ranks));
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", f"-I{os.path.dirname(HEADER)}", "-o", str(exe), str(prog)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    o = mk.mk_opts
    want = [ctypes.sizeof(o), o.comm_sms.offset, o.wait_timeout_ns.offset, o.trace.offset,
            o.trace_bytes.offset, o.num_ctas.offset, o.flags.offset, o.debug_skip_unit.offset,
            ctypes.sizeof(mk.mk_trace_record), o.raster_group.offset, o.reduce_split.offset,
            o.chain_ranks.offset]
    assert got == want


def test_constants_match_header(mk):
    """Every MK_FLAG_* bit, status code, split mode, op and dtype the header defines has the same
    value in the binding (a wrong flag bit would silently select another layout or mode)."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    flags = dict(re.findall(r"#define\s+(MK_FLAG_[A-Z0-9_]+)\s+(\d+)u", src))
    assert flags, "no MK_FLAG_ definitions found"
    for name, value in flags.items():
        assert getattr(mk, name) == int(value), name
    enums = dict(re.findall(r"\b(MK_(?:ERR|OK|SPLIT|OP|BF16|F32)[A-Z0-9_]*)\s*=\s*(\d+)", src))
    assert len(enums) >= 15
    for name, value in enums.items():
        assert getattr(mk, name) == int(value), name


def test_defaults_and_strings(mk):
    o = mk.mk_opts_default()
    assert o.split_mode == mk.MK_SPLIT_ADAPTIVE and o.debug_skip_unit == -1
    assert o.wait_timeout_ns == 2_000_000_000 and o.num_ctas == 0
    for code in range(0, 9):
        assert mk.status_string(code) not in ("", "unknown status")
    assert mk.status_string(99) == "unknown status"


def test_workspace_size_arithmetic(mk):
    # header 256 B + flags (tiles*P*4, rounded to 256) + P*tiles fp32 tiles of 128 x BN
    P, M, N, Kr = 8, 8192, 8192, 3584
    tiles = (M // 128) * (N // 256)
    flags = (tiles * P * 4 + 255) // 256 * 256
    assert mk.mk_workspace_size(mk.MK_OP_ALLREDUCE, P, M, N, Kr) == 256 + flags + P * tiles * 128 * 256 * 4
    # N <= 128 uses 128-wide tiles; ragged shapes round up to whole tiles
    assert mk.mk_workspace_size(0, 2, 128, 128, 256) == 256 + 256 + 2 * 128 * 128 * 4
    tiles = 2 * 2
    assert mk.mk_workspace_size(0, 3, 130, 264, 8) == 256 + 256 + 3 * tiles * 128 * 256 * 4
    assert mk.mk_workspace_size(mk.MK_OP_REDUCESCATTER, 8, 16384, 8192, 1024) == \
        mk.mk_workspace_size(mk.MK_OP_ALLREDUCE, 8, 16384, 8192, 1024)
    # AllGather + GEMM: header + one flag per 128-row chunk (rounded up to pair tiles)
    assert mk.mk_workspace_size(mk.MK_OP_ALLGATHER_GEMM, 4, 512, 128, 64) == 256 + 256
    assert mk.mk_workspace_size(0, 0, 128, 128, 64) == 0
    assert mk.mk_workspace_size(0, 17, 128, 128, 64) == 0
    assert mk.mk_workspace_size(0, 2, -1, 128, 64) == 0


FAKE = 0x10000  # 16-byte aligned host-side stand-in; never dereferenced by the checks below


def call_ar(mk, P=2, M=128, N=128, Kr=64, A=None, B=None, C=None, ws=FAKE, ws_bytes=None, dtype=0,
            opts=None):
    A = [FAKE] * P if A is None else A
    B = [FAKE] * P if B is None else B
    C = [FAKE] * P if C is None else C
    nb = mk.mk_workspace_size(0, max(P, 1), max(M, 0), max(N, 0), max(Kr, 0)) if ws_bytes is None else ws_bytes
    return mk.mk_gemm_allreduce(P, M, N, Kr, A, B, C, dtype, ws, ws_bytes=nb, opts=opts, stream=0)


def test_argument_checks_return_before_any_launch(mk):
    assert call_ar(mk, P=0) == mk.MK_ERR_INVALID_ARG
    assert call_ar(mk, P=17, A=[FAKE] * 17, B=[FAKE] * 17, C=[FAKE] * 17) == mk.MK_ERR_INVALID_ARG
    assert call_ar(mk, M=-1) == mk.MK_ERR_INVALID_ARG
    assert call_ar(mk, dtype=7) == mk.MK_ERR_INVALID_ARG
    assert call_ar(mk, ws=0) == mk.MK_ERR_INVALID_ARG
    assert call_ar(mk, N=100) == mk.MK_ERR_UNSUPPORTED_SHAPE
    assert call_ar(mk, Kr=60) == mk.MK_ERR_UNSUPPORTED_SHAPE
    assert call_ar(mk, A=[FAKE, FAKE + 8]) == mk.MK_ERR_ALIGNMENT
    assert call_ar(mk, C=[FAKE, 0]) == mk.MK_ERR_INVALID_ARG
    assert call_ar(mk, ws=FAKE + 128) == mk.MK_ERR_ALIGNMENT
    assert call_ar(mk, ws_bytes=1024) == mk.MK_ERR_WORKSPACE_TOO_SMALL
    o = mk.mk_opts_default()
    o.split_mode = 5
    assert call_ar(mk, opts=o) == mk.MK_ERR_INVALID_ARG
    o = mk.mk_opts_default()
    o.split_mode = mk.MK_SPLIT_STATIC
    o.comm_sms = 0
    assert call_ar(mk, opts=o) == mk.MK_ERR_INVALID_ARG
    for bad in (-1, 65):
        o = mk.mk_opts_default()
        o.reduce_split = bad
        assert call_ar(mk, opts=o) == mk.MK_ERR_INVALID_ARG and "reduce_split" in mk.mk_last_error()
    for bad in (-1, 17):
        o = mk.mk_opts_default()
        o.chain_ranks = bad
        assert call_ar(mk, opts=o) == mk.MK_ERR_INVALID_ARG and "chain_ranks" in mk.mk_last_error()
    assert call_ar(mk, N=100) == mk.MK_ERR_UNSUPPORTED_SHAPE and "multiples of 8" in mk.mk_last_error()
    # bf16 partial tiles need a split that stores partial tiles
    for mode in (mk.MK_SPLIT_ACCUMULATE, mk.MK_SPLIT_CHAINED):
        o = mk.mk_opts_default()
        o.split_mode = mode
        o.flags = mk.MK_FLAG_BF16_PARTIALS
        assert call_ar(mk, opts=o) == mk.MK_ERR_INVALID_ARG and "BF16_PARTIALS" in mk.mk_last_error()
    o = mk.mk_opts_default()
    o.flags = mk.MK_FLAG_BF16_PARTIALS
    st = mk.mk_allgather_gemm(2, 256, 128, 64, [FAKE] * 2, [FAKE] * 2, [FAKE] * 2, [FAKE] * 2, mk.MK_BF16, FAKE,
                              ws_bytes=1 << 30, opts=o, stream=0)
    assert st == mk.MK_ERR_INVALID_ARG and "BF16_PARTIALS" in mk.mk_last_error()
    # B given as N x K_r is for the row-parallel ops only
    o = mk.mk_opts_default()
    o.flags = mk.MK_FLAG_B_NK
    st = mk.mk_allgather_gemm(2, 256, 128, 64, [FAKE] * 2, [FAKE] * 2, [FAKE] * 2, [FAKE] * 2, mk.MK_BF16, FAKE,
                              ws_bytes=1 << 30, opts=o, stream=0)
    assert st == mk.MK_ERR_INVALID_ARG and "B_NK" in mk.mk_last_error()
    # ReduceScatter needs M divisible by P
    st = mk.mk_gemm_reducescatter(3, 128, 128, 64, [FAKE] * 3, [FAKE] * 3, [FAKE] * 3, 0, FAKE,
                                  ws_bytes=1 << 30, stream=0)
    assert st == mk.MK_ERR_UNSUPPORTED_SHAPE


def test_empty_problem_is_a_no_op(mk):
    # M == 0 or N == 0: validated, then nothing to launch
    assert call_ar(mk, M=0) == mk.MK_OK
    assert call_ar(mk, N=0) == mk.MK_OK


def call_attn(mk, P=2, H=2, S=256, d=128, Q=None, K=None, V=None, O=None, lse=None, ring=None, dtype=0, scale=0.0,
              ws=FAKE, ws_bytes=1 << 30, opts=None):
    Q = Q if Q is not None else [FAKE] * P
    K = K if K is not None else [FAKE] * P
    V = V if V is not None else [FAKE] * P
    O = O if O is not None else [FAKE] * P
    return mk.mk_ring_attention(P, H, S, d, Q, K, V, O, lse, ring, dtype, scale, ws, ws_bytes=ws_bytes, opts=opts,
                                stream=0)


def test_ring_attention_argument_checks_return_before_any_launch(mk):
    assert call_attn(mk, P=0) == mk.MK_ERR_INVALID_ARG
    assert call_attn(mk, P=17, Q=[FAKE] * 17, K=[FAKE] * 17, V=[FAKE] * 17, O=[FAKE] * 17) == mk.MK_ERR_INVALID_ARG
    assert call_attn(mk, S=-1) == mk.MK_ERR_INVALID_ARG
    assert call_attn(mk, dtype=3) == mk.MK_ERR_INVALID_ARG
    assert call_attn(mk, scale=-1.0) == mk.MK_ERR_INVALID_ARG
    assert call_attn(mk, d=64) == mk.MK_ERR_UNSUPPORTED_SHAPE and "head dimension" in mk.mk_last_error()
    assert call_attn(mk, ws=0) == mk.MK_ERR_INVALID_ARG
    assert call_attn(mk, Q=[FAKE, 0]) == mk.MK_ERR_INVALID_ARG
    assert call_attn(mk, V=[FAKE, FAKE + 8]) == mk.MK_ERR_ALIGNMENT
    assert call_attn(mk, lse=[FAKE, 0]) == mk.MK_ERR_INVALID_ARG
    assert call_attn(mk, ring=[FAKE, 0]) == mk.MK_ERR_INVALID_ARG
    assert call_attn(mk, ring=[FAKE, FAKE + 4]) == mk.MK_ERR_ALIGNMENT
    assert call_attn(mk, ws=FAKE + 64) == mk.MK_ERR_ALIGNMENT
    assert call_attn(mk, ws_bytes=256) == mk.MK_ERR_WORKSPACE_TOO_SMALL
    for mode in (mk.MK_SPLIT_ACCUMULATE, mk.MK_SPLIT_CHAINED):
        o = mk.mk_opts_default()
        o.split_mode = mode
        assert call_attn(mk, opts=o) == mk.MK_ERR_INVALID_ARG
    for flag in (mk.MK_FLAG_BF16_PARTIALS, mk.MK_FLAG_B_NK):
        o = mk.mk_opts_default()
        o.flags = flag
        assert call_attn(mk, opts=o) == mk.MK_ERR_INVALID_ARG
    # nothing to compute: validated, then no launch
    assert call_attn(mk, H=0) == mk.MK_OK
    assert call_attn(mk, S=0) == mk.MK_OK


def test_ring_attention_workspace_size(mk):
    # header, then one 32-bit readiness flag per forwarded 128-row KV tile: P * (P-1) * H * ceil(S/128)
    for P, H, S in ((2, 2, 256), (8, 32, 4096), (3, 5, 130), (1, 4, 1000)):
        n = P * (P - 1) * H * ((S + 127) // 128)
        want = 256 + ((max(n, 1) * 4 + 255) // 256) * 256
        assert mk.mk_ring_attention_workspace_size(P, H, S, 128) == want
    assert mk.mk_ring_attention_workspace_size(0, 1, 1, 128) == 0
    assert mk.mk_ring_attention_workspace_size(2, -1, 1, 128) == 0
