"""Fused MoE expert GEMM + EP-combine send for GB300 (sm_103a).

Python binding of the C ABI in ``include/moe_ep.h`` (``libmoe_ep.so``), with the
same entry-point names. It only marshals arguments: pointers are plain integers
(or objects with ``data_ptr()``), streams are ``cudaStream_t`` handles (or
objects with ``cuda_stream``). Every step of the path runs in the library's
kernels; there is no fallback, and a missing library raises.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH, build  # noqa: F401

EP_MAX_RANKS = 8
EP_MAX_LOCAL_EXPERTS = 256

EP_OK = 0
EP_ERR_INVALID_ARG = -1
EP_ERR_UNSUPPORTED = -2
EP_ERR_CUDA = -3

EP_STATUS_BOUNDS = 0x1
EP_STATUS_TIMEOUT = 0x2
EP_STATUS_CAPACITY = 0x4
EP_ACT_NONE = 0
EP_ACT_SWIGLU = 1
EP_SIGNAL_RANK_FLAG = 0
EP_SIGNAL_PER_EXPERT = 1
EP_OVERLAP_NONE = 0
EP_OVERLAP_ANY = 1
EP_OVERLAP_INPUTS_READY = 2
EP_STATUS_ROUTING = 0x8
EP_STATUS_INTERNAL = 0x10

EP_BF16 = 0
EP_FP8_1D2D = 1

_c_i32, _c_i64, _c_u64, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p


class ep_config(ctypes.Structure):
    _fields_ = [(n, _c_i32) for n in ("n_ranks", "my_rank", "n_local_experts", "top_k",
                                      "num_tokens", "max_tokens_per_rank", "K", "N",
                                      "msg_bytes", "dtype", "send_warps", "signal_mode")]


class ep_plan_out(ctypes.Structure):
    _fields_ = [("expert_offsets", _vp), ("src_info", _vp), ("seg_offsets", _vp),
                ("send_counts", _vp), ("gather_idx", _vp), ("m_total", _vp), ("status", _vp),
                ("max_rows", _c_i64)]


class ep_send_args(ctypes.Structure):
    _fields_ = [("A", _vp), ("a_scales", _vp), ("W", _vp), ("w_scales", _vp),
                ("expert_offsets", _vp), ("src_info", _vp), ("seg_offsets", _vp),
                ("send_counts", _vp), ("max_rows", _c_i64),
                ("recv_buf_ptrs", _vp * EP_MAX_RANKS), ("recv_count_ptrs", _vp * EP_MAX_RANKS),
                ("atomic_counter", _vp), ("rank_completion_counter", _vp), ("epoch", _c_u64),
                ("p3_control", _c_i32), ("C", _vp), ("status", _vp), ("trace", _vp),
                ("timeout_ns", _c_i64), ("trace_records", _c_i64),
                ("local_activation", _c_i32), ("overlap_previous", _c_i32)]


class ep_combine_args(ctypes.Structure):
    _fields_ = [("recv_buf", _vp), ("recv_count", _vp), ("gates", _vp), ("out", _vp),
                ("epoch", _c_u64), ("timeout_ns", _c_i64), ("status", _vp),
                ("topk_ids", _vp), ("overlap_previous", _c_i32)]


class ep_scatter_args(ctypes.Structure):
    _fields_ = [("C", _vp), ("expert_offsets", _vp), ("src_info", _vp), ("seg_offsets", _vp),
                ("send_counts", _vp), ("max_rows", _c_i64),
                ("recv_buf_ptrs", _vp * EP_MAX_RANKS), ("recv_count_ptrs", _vp * EP_MAX_RANKS),
                ("block_counter", _vp), ("epoch", _c_u64), ("status", _vp)]


class ep_dispatch_args(ctypes.Structure):
    _fields_ = [("x_ptrs", _vp * EP_MAX_RANKS), ("gather_idx", _vp), ("expert_offsets", _vp),
                ("max_rows", _c_i64), ("hidden", _c_i32), ("A_in", _vp), ("status", _vp)]


class ep_swiglu_args(ctypes.Structure):
    _fields_ = [("G", _vp), ("A", _vp), ("expert_offsets", _vp), ("max_rows", _c_i64),
                ("inter", _c_i32)]


EP_IPC_HANDLE_BYTES = 64


class ep_ipc_handle(ctypes.Structure):
    _fields_ = [("handle", ctypes.c_uint8 * EP_IPC_HANDLE_BYTES), ("offset", _c_u64),
                ("bytes", _c_u64)]


class EpError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {ep_strerror(code)} ({code})")
        self.code = code


_lib = None

EXPORTS = ("ep_plan_sizes", "ep_plan", "grouped_gemm_combine_send", "ep_combine_reduce",
           "ep_strerror", "grouped_gemm_combine_send_noalloc", "ep_scatter_send",
           "ep_dispatch_gather", "ep_swiglu", "ep_ipc_export", "ep_ipc_import", "ep_ipc_close")


def load(build_if_missing: bool = True):
    """Load libmoe_ep.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        build()
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} not built; run moe_expert_gemm_gb300.build()")
    L = ctypes.CDLL(LIB_PATH)
    L.ep_plan_sizes.argtypes = [ctypes.POINTER(ep_config), ctypes.POINTER(_c_i64)]
    L.ep_plan.argtypes = [ctypes.POINTER(ep_config), _vp, ctypes.POINTER(ep_plan_out), _vp]
    L.grouped_gemm_combine_send.argtypes = [ctypes.POINTER(ep_config),
                                            ctypes.POINTER(ep_send_args), _vp]
    L.ep_combine_reduce.argtypes = [ctypes.POINTER(ep_config), ctypes.POINTER(ep_combine_args),
                                    _vp]
    L.grouped_gemm_combine_send_noalloc.argtypes = [ctypes.POINTER(ep_config),
                                                    ctypes.POINTER(ep_send_args), _vp]
    L.ep_scatter_send.argtypes = [ctypes.POINTER(ep_config), ctypes.POINTER(ep_scatter_args), _vp]
    L.ep_dispatch_gather.argtypes = [ctypes.POINTER(ep_config), ctypes.POINTER(ep_dispatch_args),
                                     _vp]
    L.ep_swiglu.argtypes = [ctypes.POINTER(ep_config), ctypes.POINTER(ep_swiglu_args), _vp]
    L.ep_ipc_export.argtypes = [_vp, ctypes.POINTER(ep_ipc_handle)]
    L.ep_ipc_import.argtypes = [ctypes.POINTER(ep_ipc_handle), ctypes.POINTER(_vp)]
    L.ep_ipc_close.argtypes = [ctypes.POINTER(ep_ipc_handle), _vp]
    for f in ("ep_plan_sizes", "ep_plan", "grouped_gemm_combine_send", "ep_combine_reduce",
              "grouped_gemm_combine_send_noalloc", "ep_scatter_send", "ep_dispatch_gather",
              "ep_swiglu", "ep_ipc_export", "ep_ipc_import", "ep_ipc_close"):
        getattr(L, f).restype = ctypes.c_int
    L.ep_strerror.argtypes = [ctypes.c_int]
    L.ep_strerror.restype = ctypes.c_char_p
    _lib = L
    return L


def ptr(x) -> int:
    """Device address of a tensor-like object, or the integer itself (None -> 0)."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def stream_handle(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(rc: int, where: str) -> int:
    if rc != EP_OK:
        raise EpError(rc, where)
    return rc


def ep_strerror(code: int) -> str:
    return load().ep_strerror(code).decode()


def ep_plan_sizes(cfg: ep_config) -> int:
    out = _c_i64(0)
    _check(load().ep_plan_sizes(ctypes.byref(cfg), ctypes.byref(out)), "ep_plan_sizes")
    return int(out.value)


def ep_plan(cfg: ep_config, topk_ids, out: ep_plan_out, stream=None) -> int:
    return _check(load().ep_plan(ctypes.byref(cfg), ptr(topk_ids), ctypes.byref(out),
                                 stream_handle(stream)), "ep_plan")


def grouped_gemm_combine_send(cfg: ep_config, args: ep_send_args, stream=None) -> int:
    return _check(load().grouped_gemm_combine_send(ctypes.byref(cfg), ctypes.byref(args),
                                                   stream_handle(stream)),
                  "grouped_gemm_combine_send")


def grouped_gemm_combine_send_noalloc(cfg: ep_config, args: ep_send_args, stream=None) -> int:
    """The fused send for callers that cannot allocate: the counter arrays come
    from the library's own device array (args' counter pointers are ignored)."""
    return _check(load().grouped_gemm_combine_send_noalloc(ctypes.byref(cfg), ctypes.byref(args),
                                                           stream_handle(stream)),
                  "grouped_gemm_combine_send_noalloc")


def ep_scatter_send(cfg: ep_config, args: ep_scatter_args, stream=None) -> int:
    """The send step alone (unfused comparator): local C rows to the receive
    buffers, then the count words and the rank flags."""
    return _check(load().ep_scatter_send(ctypes.byref(cfg), ctypes.byref(args),
                                         stream_handle(stream)), "ep_scatter_send")


def ep_dispatch_gather(cfg: ep_config, args: ep_dispatch_args, stream=None) -> int:
    """Dispatch: every routed token row to its expert's rank, in plan order."""
    return _check(load().ep_dispatch_gather(ctypes.byref(cfg), ctypes.byref(args),
                                            stream_handle(stream)), "ep_dispatch_gather")


def ep_swiglu(cfg: ep_config, args: ep_swiglu_args, stream=None) -> int:
    """A = bf16(SiLU(gate) * up) from the up/gate GEMM's rows."""
    return _check(load().ep_swiglu(ctypes.byref(cfg), ctypes.byref(args),
                                   stream_handle(stream)), "ep_swiglu")


def ep_combine_reduce(cfg: ep_config, args: ep_combine_args, stream=None) -> int:
    return _check(load().ep_combine_reduce(ctypes.byref(cfg), ctypes.byref(args),
                                           stream_handle(stream)), "ep_combine_reduce")


def ep_ipc_export(dev_ptr) -> ep_ipc_handle:
    """CUDA IPC handle (plus offset) of a device buffer of this process, for the peer
    processes of an expert-parallel group to map (ep_ipc_import)."""
    h = ep_ipc_handle()
    _check(load().ep_ipc_export(ptr(dev_ptr), ctypes.byref(h)), "ep_ipc_export")
    return h


def ep_ipc_import(h: ep_ipc_handle) -> int:
    """Map another process's exported buffer; returns its address in this process."""
    out = _vp(0)
    _check(load().ep_ipc_import(ctypes.byref(h), ctypes.byref(out)), "ep_ipc_import")
    return int(out.value)


def ep_ipc_close(h: ep_ipc_handle, dev_ptr: int) -> int:
    return _check(load().ep_ipc_close(ctypes.byref(h), ptr(dev_ptr)), "ep_ipc_close")


def raw_call(name: str, *args) -> int:
    """Call an entry point and return its code without raising (for error-path tests)."""
    return int(getattr(load(), name)(*args))
