"""Oracle for the fused MoE expert GEMM + EP-combine path -- TEST INFRASTRUCTURE.

A plain CPU restatement (C in ``moe_oracle.c``, loaded with ctypes) of what the
path computes, following the pages "EpiloguePeerSink" (send_tile: the finished
tile goes to the token-owning peers instead of the local store),
"P3PeerSendConfig" (description: recv_count_layout and recv_buf_layout) and
"ep_signal_completion" (per-expert counts, acquire-release election, rank flag).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA path.

Every function here is pinned by ``tests/test_oracle_pins.py`` to something
other than itself (library routines, closed forms, brute force, special cases);
the one unpinned aspect is the order of floating-point accumulation, which the
pages do not fix and which only matters below the stated tolerances.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmoe_oracle.so")

BF16, FP8_1D2D = 0, 1

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no vendor code, no BLAS)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        i32, i64, u64, vp, f64 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                  ctypes.c_void_p, ctypes.c_double)
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_double.restype = f64
        L.orc_bf16_from_double.argtypes = [f64]
        L.orc_bf16_from_double.restype = ctypes.c_uint16
        L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_to_double.restype = f64
        for name in ("orc_bf16_to_double_n", "orc_bf16_from_double_n", "orc_e4m3_to_double_n"):
            getattr(L, name).argtypes = [vp, vp, i64]
            getattr(L, name).restype = None
        L.orc_recv_count_index.argtypes = [i64, i64, i64]
        L.orc_recv_count_index.restype = i64
        L.orc_recv_buf_offset.argtypes = [i64, i64, i64, i64, i64]
        L.orc_recv_buf_offset.restype = i64
        L.orc_plan.argtypes = [ctypes.c_int] * 5 + [vp, i64] + [vp] * 6
        L.orc_plan.restype = ctypes.c_int
        L.orc_expert_rows.argtypes = ([ctypes.c_int, vp, vp, vp, vp, vp] + [ctypes.c_int] * 3
                                      + [vp, i64, vp, ctypes.c_int])
        L.orc_expert_rows.restype = ctypes.c_int
        L.orc_expert_rows2.argtypes = ([ctypes.c_int, vp, vp, vp, vp, vp] + [ctypes.c_int] * 3
                                       + [vp, i64, vp, vp, ctypes.c_int])
        L.orc_expert_rows2.restype = ctypes.c_int
        L.orc_combine_exact.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, i64, vp]
        L.orc_combine_exact.restype = None
        L.orc_scatter.argtypes = ([vp, vp, i64, ctypes.c_int, vp, vp, vp] + [ctypes.c_int] * 3
                                  + [i64, i64, vp, vp])
        L.orc_scatter.restype = i64
        L.orc_signal.argtypes = [ctypes.c_int] * 3 + [vp, u64, vp, vp, vp]
        L.orc_signal.restype = ctypes.c_int
        L.orc_combine.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, i64, vp, i64, vp,
                                  ctypes.c_int]
        L.orc_combine.restype = None
        _lib = L
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


# ------------------------------------------------------------------ formats

def bf16_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().orc_bf16_to_double_n(_p(b), _p(out), b.size)
    return out


def bf16_from_f64(x) -> np.ndarray:
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_bf16_from_double_n(_p(v), _p(out), v.size)
    return out


def e4m3_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    lib().orc_e4m3_to_double_n(_p(b), _p(out), b.size)
    return out


def recv_count_index(e: int, rk: int, n_ranks: int) -> int:
    return lib().orc_recv_count_index(e, rk, n_ranks)


def recv_buf_offset(src_idx: int, src_topk: int, byte_off: int, top_k: int, msg_bytes: int) -> int:
    return lib().orc_recv_buf_offset(src_idx, src_topk, byte_off, top_k, msg_bytes)


# --------------------------------------------------------------------- plan

@dataclass
class Plan:
    expert_offsets: np.ndarray  # int32 [El+1]
    src_info: np.ndarray  # int32 [m_total, 2]
    seg_offsets: np.ndarray  # int32 [El, R+1]
    send_counts: np.ndarray  # int32 [El, R]
    gather_idx: np.ndarray  # int32 [m_total]
    m_total: int


def plan(n_ranks: int, n_local_experts: int, top_k: int, topk_ids: np.ndarray, rank: int,
         max_rows: int | None = None) -> Plan:
    R, El, k = n_ranks, n_local_experts, top_k
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T = ids.shape[1]
    assert ids.shape == (R, T, k)
    if max_rows is None:
        max_rows = R * T * min(k, El)
    eo = np.zeros(El + 1, np.int32)
    si = np.zeros((max(max_rows, 1), 2), np.int32)
    seg = np.zeros((El, R + 1), np.int32)
    sc = np.zeros((El, R), np.int32)
    gi = np.zeros(max(max_rows, 1), np.int32)
    mt = np.zeros(1, np.int32)
    rc = lib().orc_plan(R, El, T, k, rank, _p(ids), max_rows, _p(eo), _p(si), _p(seg), _p(sc),
                        _p(gi), _p(mt))
    if rc != 0:
        raise ValueError({-1: "rows exceed max_rows", -2: "expert id out of range"}.get(rc, rc))
    m = int(mt[0])
    return Plan(eo, si[:m].copy(), seg, sc, gi[:m].copy(), m)


# ------------------------------------------------------------- expert rows

def expert_rows(dtype: int, A, W, expert_offsets, K: int, N: int, rows=None, a_scales=None,
                w_scales=None, threads: int | None = None, exact: bool = False):
    """bf16 bit patterns [len(rows), N] of the down-projection rows requested;
    with ``exact`` a pair (bf16 bits, unrounded float64 sums)."""
    El = len(expert_offsets) - 1
    eo = np.ascontiguousarray(expert_offsets, dtype=np.int32)
    if rows is None:
        rows = np.arange(int(eo[-1]), dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if dtype == BF16:
        A = np.ascontiguousarray(A, dtype=np.uint16)
        W = np.ascontiguousarray(W, dtype=np.uint16)
        sa = sw = None
    else:
        A = np.ascontiguousarray(A, dtype=np.uint8)
        W = np.ascontiguousarray(W, dtype=np.uint8)
        sa = np.ascontiguousarray(a_scales, dtype=np.float32)
        sw = np.ascontiguousarray(w_scales, dtype=np.float32)
    Y = np.zeros((len(rows), N), np.uint16)
    Yd = np.zeros((len(rows), N), np.float64) if exact else None
    if len(rows):
        rc = lib().orc_expert_rows2(dtype, _p(A), None if sa is None else _p(sa), _p(W),
                                    None if sw is None else _p(sw), _p(eo), El, K, N, _p(rows),
                                    len(rows), _p(Y), None if Yd is None else _p(Yd),
                                    threads or default_threads())
        if rc != 0:
            raise ValueError(f"orc_expert_rows failed: {rc}")
    return (Y, Yd) if exact else Y


# ------------------------------------------------------------------ scatter

def scatter(Y, rows, pl: Plan, n_ranks: int, top_k: int, N: int, msg_bytes: int,
            max_tokens: int, recv_bufs: list, hits: np.ndarray | None = None):
    """Write rows into the receive buffers (a list of uint8 arrays, one per rank).
    Returns (hits [R, max_tokens*top_k], number of out-of-bounds rows)."""
    R = n_ranks
    El = len(pl.expert_offsets) - 1
    Y = np.ascontiguousarray(Y, dtype=np.uint16)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if hits is None:
        hits = np.zeros((R, max_tokens * top_k), np.int32)
    ptrs = (ctypes.c_void_p * R)(*[b.ctypes.data for b in recv_bufs])
    si = np.ascontiguousarray(pl.src_info, dtype=np.int32)
    if si.size == 0:
        si = np.zeros((1, 2), np.int32)
    bad = lib().orc_scatter(_p(Y), _p(rows), len(rows), N, _p(pl.expert_offsets), _p(si),
                            _p(pl.seg_offsets), El, R, top_k, msg_bytes, max_tokens,
                            ctypes.cast(ptrs, ctypes.c_void_p), _p(hits))
    return hits, int(bad)


# --------------------------------------------------------------- signalling

def signal(n_ranks: int, n_local_experts: int, rank: int, send_counts, epoch: int,
           recv_counts: list, rank_counter: np.ndarray) -> np.ndarray:
    """Run one producer rank's completion signalling; returns the event log
    [n_events, 4] = (kind 0 count / 1 flag, expert, dst, old counter)."""
    R, El = n_ranks, n_local_experts
    sc = np.ascontiguousarray(send_counts, dtype=np.int32)
    ptrs = (ctypes.c_void_p * R)(*[b.ctypes.data for b in recv_counts])
    log = np.zeros((El * R + R, 4), np.int32)
    n = lib().orc_signal(R, El, rank, _p(sc), epoch, ctypes.cast(ptrs, ctypes.c_void_p),
                         _p(rank_counter), _p(log))
    return log[:n].copy()


def signal_per_expert(n_ranks: int, n_local_experts: int, rank: int, send_counts, epoch: int,
                      recv_counts: list) -> np.ndarray:
    """The default ("not ep_ord_r") mode of "ep_signal_completion": every expert's
    count word is its own arrival signal, so it must tell this call from the last
    one: word e*R + rank of every destination's count buffer becomes
    (epoch mod 2^32) << 32 | rows; the rank-flag words are not written and there
    is no election. Returns the event log [El*R, 4] = (0, expert, dst, 0)."""
    R, El = n_ranks, n_local_experts
    sc = np.asarray(send_counts, dtype=np.int64).reshape(El, R)
    tag = (int(epoch) & 0xFFFFFFFF) << 32
    log = []
    for e in range(El):
        for dst in range(R):
            recv_counts[dst][e * R + rank] = np.uint64(tag | int(sc[e, dst]))
            log.append((0, e, dst, 0))
    return np.array(log, np.int32).reshape(-1, 4)


# ------------------------------------------------------------ layer steps

def dispatch(pl: Plan, tokens: list, top_k: int) -> np.ndarray:
    """The dispatch step before the down-projection's path: row m of the plan,
    (source rank rk, token t, slot j) = gather_idx[m] = (rk*T + t)*top_k + j,
    receives token row tokens[rk][t] unchanged (bf16 bit patterns)."""
    T = tokens[0].shape[0]
    out = np.zeros((pl.m_total, tokens[0].shape[1]), np.uint16)
    for m in range(pl.m_total):
        gi = int(pl.gather_idx[m])
        rk, t = gi // (T * top_k), (gi % (T * top_k)) // top_k
        out[m] = tokens[rk][t]
    return out


def swiglu(G_bits: np.ndarray, inter: int) -> np.ndarray:
    """The gated activation: A[m][i] = bf16(SiLU(G[m][i]) * G[m][inter + i]) with
    SiLU(x) = x / (1 + e^-x), evaluated in float64 on the bf16 values of G and
    rounded to nearest even once."""
    g = bf16_to_f64(np.ascontiguousarray(G_bits[:, :inter]))
    u = bf16_to_f64(np.ascontiguousarray(G_bits[:, inter:2 * inter]))
    return bf16_from_f64(g / (1.0 + np.exp(-g)) * u)


def swiglu_exact(G: np.ndarray, inter: int) -> np.ndarray:
    """The same activation applied to the unrounded (float64) products, as the
    up/gate projection with the activation in its epilogue computes it: the gate
    and up values are never rounded to bf16, only the result is."""
    g, u = G[:, :inter], G[:, inter:2 * inter]
    return bf16_from_f64(g / (1.0 + np.exp(-g)) * u)


# ------------------------------------------------------------------ combine

def combine(recv_buf, gates, top_k: int, N: int, msg_bytes: int, tokens=None,
            threads: int | None = None) -> np.ndarray:
    """bf16 bit patterns [len(tokens), N] of the gate-weighted combine."""
    recv = np.ascontiguousarray(recv_buf, dtype=np.uint8)
    g = np.ascontiguousarray(gates, dtype=np.float32)
    T = g.shape[0]
    if tokens is None:
        tokens = np.arange(T, dtype=np.int64)
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    out = np.zeros((len(tokens), N), np.uint16)
    if len(tokens):
        lib().orc_combine(_p(recv), _p(g), top_k, N, msg_bytes, _p(tokens), len(tokens),
                          _p(out), threads or default_threads())
    return out


def combine_exact(rows_f64, gates) -> np.ndarray:
    """Exact gate-weighted sums [n, N] of exact rows [n, k, N] (float64, unrounded)."""
    y = np.ascontiguousarray(rows_f64, dtype=np.float64)
    g = np.ascontiguousarray(gates, dtype=np.float32)
    n, k, N = y.shape
    out = np.zeros((n, N), np.float64)
    lib().orc_combine_exact(_p(y), _p(g), k, N, n, _p(out))
    return out


from .pipeline import full_pipeline, sampled_pipeline  # noqa: E402,F401
