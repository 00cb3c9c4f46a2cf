"""Thin ctypes binding of libmk.so (include/mk.h).  Argument marshalling only.

Every entry point of the C ABI is exposed under its own name and takes the same arguments;
pointer arrays may be given as lists of torch tensors or of integer device addresses, and the
stream as a torch.cuda.Stream, an integer handle or None (the current torch stream).  The
computation always runs in libmk.so; if the library is missing this module raises on import.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmk.so")

MK_OK = 0
MK_ERR_INVALID_ARG = 1
MK_ERR_UNSUPPORTED_SHAPE = 2
MK_ERR_ALIGNMENT = 3
MK_ERR_WORKSPACE_TOO_SMALL = 4
MK_ERR_CUDA = 5
MK_ERR_TIMEOUT = 6
MK_ERR_INTERNAL = 7
MK_ERR_NOT_RESIDENT = 8

MK_BF16 = 0
MK_F32 = 1

MK_OP_ALLREDUCE = 0
MK_OP_REDUCESCATTER = 1
MK_OP_ALLGATHER_GEMM = 2

MK_SPLIT_ADAPTIVE = 0
MK_SPLIT_STATIC = 1
MK_SPLIT_UNFUSED = 2
MK_SPLIT_ACCUMULATE = 3
MK_SPLIT_CHAINED = 4

MK_FLAG_KEEP_PARTIALS = 1
MK_FLAG_SINGLE_SM_TILES = 2
MK_FLAG_NO_L2_HINTS = 4
MK_FLAG_NO_COOPERATIVE = 8
MK_FLAG_TILE_MAJOR = 16
MK_FLAG_RANK_MAJOR = 32
MK_FLAG_NO_EPILOGUE_PACING = 64
MK_FLAG_BF16_PARTIALS = 128
MK_FLAG_B_NK = 256

# Every extern "C" symbol declared in include/mk.h.
EXPORTED = ("mk_opts_default", "mk_workspace_size", "mk_gemm_allreduce", "mk_gemm_reducescatter",
            "mk_allgather_gemm", "mk_ring_attention_workspace_size", "mk_ring_attention",
            "mk_gemm_allreduce_noalloc", "mk_status_check", "mk_status_string", "mk_last_error")

MK_NOALLOC_MAX_WS_BYTES = 64 << 20


class mk_opts(ctypes.Structure):
    _fields_ = [("split_mode", ctypes.c_int32), ("comm_sms", ctypes.c_int32),
                ("wait_timeout_ns", ctypes.c_uint64), ("trace", ctypes.c_void_p),
                ("trace_bytes", ctypes.c_uint64), ("num_ctas", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("debug_skip_unit", ctypes.c_int64),
                ("raster_group", ctypes.c_int32), ("reduce_split", ctypes.c_int32),
                ("chain_ranks", ctypes.c_int32)]


class mk_trace_record(ctypes.Structure):
    _fields_ = [("t_ns", ctypes.c_uint64), ("target", ctypes.c_uint32),
                ("units_done", ctypes.c_uint32), ("tiles_done", ctypes.c_uint32),
                ("num_blocks", ctypes.c_uint32), ("reserved", ctypes.c_uint64)]


class MkError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"mk status {status} ({status_string(status)}): {detail}")
        self.status = status


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run gemm_tile_level_gb300.build.build() "
                      "(or __graft_entry__.build()) first")

_lib = ctypes.CDLL(LIB_PATH)
_vp, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
_PP = ctypes.POINTER(ctypes.c_void_p)
_lib.mk_opts_default.argtypes = [ctypes.POINTER(mk_opts)]
_lib.mk_opts_default.restype = None
_lib.mk_workspace_size.argtypes = [_i32, _i32, _i64, _i64, _i64]
_lib.mk_workspace_size.restype = ctypes.c_size_t
for _name in ("mk_gemm_allreduce", "mk_gemm_reducescatter"):
    getattr(_lib, _name).argtypes = [_i32, _i64, _i64, _i64, _PP, _PP, _PP, _i32, _vp,
                                     ctypes.c_size_t, ctypes.POINTER(mk_opts), _vp]
    getattr(_lib, _name).restype = _i32
_lib.mk_allgather_gemm.argtypes = [_i32, _i64, _i64, _i64, _PP, _PP, _PP, _PP, _i32, _vp,
                                   ctypes.c_size_t, ctypes.POINTER(mk_opts), _vp]
_lib.mk_allgather_gemm.restype = _i32
_lib.mk_ring_attention_workspace_size.argtypes = [_i32, _i64, _i64, _i64]
_lib.mk_ring_attention_workspace_size.restype = ctypes.c_size_t
_lib.mk_ring_attention.argtypes = [_i32, _i64, _i64, _i64, _PP, _PP, _PP, _PP, _PP, _PP, _i32, ctypes.c_float, _vp,
                                   ctypes.c_size_t, ctypes.POINTER(mk_opts), _vp]
_lib.mk_ring_attention.restype = _i32
_lib.mk_gemm_allreduce_noalloc.argtypes = [_i32, _i64, _i64, _i64, _PP, _PP, _PP, _i32,
                                           ctypes.POINTER(mk_opts), _vp]
_lib.mk_gemm_allreduce_noalloc.restype = _i32
_lib.mk_status_check.argtypes = [_vp, _vp]
_lib.mk_status_check.restype = _i32
_lib.mk_status_string.argtypes = [_i32]
_lib.mk_status_string.restype = ctypes.c_char_p
_lib.mk_last_error.argtypes = []
_lib.mk_last_error.restype = ctypes.c_char_p


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptrs(xs):
    if xs is None:
        return None
    return (ctypes.c_void_p * len(xs))(*[_addr(x) for x in xs])


def _stream(s) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _nbytes(ws) -> int:
    return int(ws.numel() * ws.element_size())


def mk_opts_default() -> mk_opts:
    o = mk_opts()
    _lib.mk_opts_default(ctypes.byref(o))
    return o


def mk_workspace_size(op: int, P: int, M: int, N: int, K_per_rank: int) -> int:
    return int(_lib.mk_workspace_size(op, P, M, N, K_per_rank))


def mk_gemm_allreduce(P, M, N, K_per_rank, A, B, C, out_dtype, ws, ws_bytes=None, opts=None,
                      stream=None) -> int:
    return int(_lib.mk_gemm_allreduce(P, M, N, K_per_rank, _ptrs(A), _ptrs(B), _ptrs(C), out_dtype,
                                      _addr(ws), _nbytes(ws) if ws_bytes is None else ws_bytes,
                                      ctypes.byref(opts) if opts is not None else None,
                                      _stream(stream)))


def mk_gemm_reducescatter(P, M, N, K_per_rank, A, B, C_shard, out_dtype, ws, ws_bytes=None,
                          opts=None, stream=None) -> int:
    return int(_lib.mk_gemm_reducescatter(P, M, N, K_per_rank, _ptrs(A), _ptrs(B), _ptrs(C_shard),
                                          out_dtype, _addr(ws),
                                          _nbytes(ws) if ws_bytes is None else ws_bytes,
                                          ctypes.byref(opts) if opts is not None else None,
                                          _stream(stream)))


def mk_allgather_gemm(P, M, N, K, A_shard, B, A_gathered, C, out_dtype, ws, ws_bytes=None,
                      opts=None, stream=None) -> int:
    return int(_lib.mk_allgather_gemm(P, M, N, K, _ptrs(A_shard), _ptrs(B), _ptrs(A_gathered),
                                      _ptrs(C), out_dtype, _addr(ws),
                                      _nbytes(ws) if ws_bytes is None else ws_bytes,
                                      ctypes.byref(opts) if opts is not None else None,
                                      _stream(stream)))


def mk_ring_attention_workspace_size(P: int, H: int, S: int, d: int) -> int:
    return int(_lib.mk_ring_attention_workspace_size(P, H, S, d))


def mk_ring_attention(P, H, S, d, Q, K, V, O, lse, kv_ring, out_dtype, scale, ws, ws_bytes=None, opts=None,
                      stream=None) -> int:
    """Ring Attention over P sequence slices; lse and kv_ring may be None."""
    return int(_lib.mk_ring_attention(P, H, S, d, _ptrs(Q), _ptrs(K), _ptrs(V), _ptrs(O), _ptrs(lse), _ptrs(kv_ring),
                                      out_dtype, float(scale), _addr(ws), _nbytes(ws) if ws_bytes is None else ws_bytes,
                                      ctypes.byref(opts) if opts is not None else None, _stream(stream)))


def mk_gemm_allreduce_noalloc(P, M, N, K_per_rank, A, B, C, out_dtype, opts=None, stream=None) -> int:
    """mk_gemm_allreduce with the library's static workspace (for callers that cannot allocate)."""
    return int(_lib.mk_gemm_allreduce_noalloc(P, M, N, K_per_rank, _ptrs(A), _ptrs(B), _ptrs(C), out_dtype,
                                              ctypes.byref(opts) if opts is not None else None,
                                              _stream(stream)))


def mk_status_check(ws, stream=None) -> int:
    return int(_lib.mk_status_check(_addr(ws), _stream(stream)))


def status_string(status: int) -> str:
    return _lib.mk_status_string(status).decode()


def mk_status_string(status: int) -> str:
    return status_string(status)


def mk_last_error() -> str:
    return _lib.mk_last_error().decode()


def check(status: int) -> None:
    """Raise MkError for a non-zero status, with the library's detail message."""
    if status != MK_OK:
        raise MkError(status, mk_last_error())
