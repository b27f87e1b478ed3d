"""Whole-path oracle runs -- TEST INFRASTRUCTURE (see the package docstring).

``full_pipeline`` plays every logical rank in turn: plan, expert rows, scatter
into every destination's receive buffer, completion signalling, then the
gate-weighted combine of every destination. ``sampled_pipeline`` computes the
same quantities for a few tokens of one destination only, for workloads too
large to run in full on the host.
"""

from __future__ import annotations

import numpy as np

from . import (BF16, FP8_1D2D, Plan, combine, combine_exact, default_threads, dispatch,
               expert_rows, plan, scatter, signal, signal_per_expert, swiglu)

SENTINEL_BYTE = 0xFF  # bf16 0xFFFF is a NaN: an unwritten slot cannot pass a value check
SENTINEL_WORD = np.uint64(0xFFFFFFFFFFFFFFFF)


def _dtype_code(dtype: str) -> int:
    return {"bf16": BF16, "fp8_1d2d": FP8_1D2D}[dtype]


def full_pipeline(w, routing, values: list, epoch: int = 1, threads: int | None = None,
                  per_expert: bool = False) -> dict:
    """Run every producer rank, then every destination's combine.

    ``values[r]`` is the operand dict of rank r (``synth.make_rank_values``).
    Returns plans, rows Y per producer, receive buffers / counts per destination,
    election counters per producer, signalling logs per producer, slot hit counts
    per destination, the combined outputs per destination (bf16 bits) and, as
    ``out_exact`` / ``rows_exact``, the exact combine of the exact rows (float64,
    no rounding anywhere) per destination. ``per_expert`` selects the default
    signalling mode (epoch-tagged count words, no rank flags) instead of ep_ord_r."""
    R, El, k, T, K, N = w.n_ranks, w.n_local_experts, w.top_k, w.tokens, w.K, w.N
    msg = w.msg_bytes
    dt = _dtype_code(w.dtype)
    recv = [np.full(T * k * msg, SENTINEL_BYTE, np.uint8) for _ in range(R)]
    counts = [np.full(El * R + R, SENTINEL_WORD, np.uint64) for _ in range(R)]
    hits = np.zeros((R, T * k), np.int32)
    plans, ys, logs, counters = [], [], [], []
    exact = [np.zeros((T, k, N)) for _ in range(R)]
    bad = 0
    for r in range(R):
        pl = plan(R, El, k, routing.topk_ids, r)
        v = values[r]
        Y, Yd = expert_rows(dt, v["A"], v["W"], pl.expert_offsets, K, N, rows=None,
                            a_scales=v.get("a_scales"), w_scales=v.get("w_scales"),
                            threads=threads, exact=True)
        rows = np.arange(pl.m_total, dtype=np.int64)
        for m in range(pl.m_total):  # the exact row, placed at its (dst, token, slot)
            e = int(np.searchsorted(pl.expert_offsets, m, side="right") - 1)
            dst = int(np.searchsorted(pl.seg_offsets[e], m, side="right") - 1)
            t, j = pl.src_info[m]
            exact[dst][t, j] = Yd[m]
        hits, b = scatter(Y, rows, pl, R, k, N, msg, T, recv, hits)
        bad += b
        ctr = np.zeros(R, np.int32)
        if per_expert:
            logs.append(signal_per_expert(R, El, r, pl.send_counts, epoch, counts))
        else:
            logs.append(signal(R, El, r, pl.send_counts, epoch, counts, ctr))
        counters.append(ctr)
        plans.append(pl)
        ys.append(Y)
    outs = [combine(recv[d], routing.gates[d], k, N, msg, threads=threads) for d in range(R)]
    out_exact = [combine_exact(exact[d], routing.gates[d]) for d in range(R)]
    return dict(plans=plans, Y=ys, recv=recv, counts=counts, hits=hits, bad=bad, logs=logs,
                counters=counters, out=outs, rows_exact=exact, out_exact=out_exact)


def row_of(pl: Plan, src_rank: int, expert_local: int, t: int, j: int) -> int:
    """Row of plan ``pl`` that carries routing entry (src_rank, t, j) for a local expert."""
    lo = int(pl.seg_offsets[expert_local, src_rank])
    hi = int(pl.seg_offsets[expert_local, src_rank + 1])
    seg = pl.src_info[lo:hi]
    hit = np.nonzero((seg[:, 0] == t) & (seg[:, 1] == j))[0]
    if len(hit) != 1:
        raise KeyError((src_rank, expert_local, t, j))
    return lo + int(hit[0])


def sampled_pipeline(w, routing, values_of, dst: int, tokens, plans: dict | None = None,
                     threads: int | None = None) -> dict:
    """Oracle rows and combined outputs for ``tokens`` of destination ``dst``.

    ``values_of(r)`` returns rank r's operand dict. Returns, per sampled token,
    the k received rows (bf16 bits [n, k, N]), the producer (rank, row) of each,
    the combined output (bf16 bits [n, N]), and the exact rows and exact combine
    (float64, unrounded) as ``rows_exact`` / ``out_exact``."""
    R, El, k, N = w.n_ranks, w.n_local_experts, w.top_k, w.N
    dt = _dtype_code(w.dtype)
    tokens = np.asarray(tokens, dtype=np.int64)
    plans = {} if plans is None else plans
    need: dict[int, list] = {}
    where = np.zeros((len(tokens), k, 2), np.int64)
    for i, t in enumerate(tokens):
        for j in range(k):
            g = int(routing.topk_ids[dst, t, j])
            r, e = g // El, g % El
            if r not in plans:
                plans[r] = plan(R, El, k, routing.topk_ids, r)
            m = row_of(plans[r], dst, e, int(t), j)
            where[i, j] = (r, m)
            need.setdefault(r, []).append(m)
    rows_out = np.zeros((len(tokens), k, N), np.uint16)
    rows_exact = np.zeros((len(tokens), k, N), np.float64)
    for r, ms in need.items():
        ms_u = np.unique(np.asarray(ms, dtype=np.int64))
        v = values_of(r)
        Y, Yd = expert_rows(dt, v["A"], v["W"], plans[r].expert_offsets, w.K, N, rows=ms_u,
                            a_scales=v.get("a_scales"), w_scales=v.get("w_scales"),
                            threads=threads or default_threads(), exact=True)
        pos = {int(m): i for i, m in enumerate(ms_u)}
        for i in range(len(tokens)):
            for j in range(k):
                if where[i, j, 0] == r:
                    rows_out[i, j] = Y[pos[int(where[i, j, 1])]]
                    rows_exact[i, j] = Yd[pos[int(where[i, j, 1])]]
    # combine over a compact receive buffer holding just these tokens' slots
    compact = rows_out.reshape(-1).view(np.uint8)
    g = np.ascontiguousarray(routing.gates[dst][tokens])
    out = combine(compact, g, k, N, 2 * N, threads=threads)
    return dict(tokens=tokens, rows=rows_out, where=where, out=out, plans=plans,
                rows_exact=rows_exact, out_exact=combine_exact(rows_exact, g))


def layer_pipeline(w, routing, layer_values: list, epoch: int = 1,
                   threads: int | None = None) -> dict:
    """A whole MoE layer around the down-projection (bf16): per producer rank, the
    dispatch of its routed token rows, the up/gate projection (expert_rows with
    K = H, N = 2I: rows rounded to bf16), the gated activation, then
    ``full_pipeline`` on the resulting A and the down-projection weights.
    ``layer_values[r]`` holds X, W1, W2 (``synth.make_layer_values``). Returns
    ``full_pipeline``'s dict plus the intermediates A_in, G, A per rank."""
    R, El, k = w.n_ranks, w.n_local_experts, w.top_k
    H, I = w.N, w.K
    tokens = [v["X"] for v in layer_values]
    A_in, Gs, As, values = [], [], [], []
    for r in range(R):
        pl = plan(R, El, k, routing.topk_ids, r)
        a_in = dispatch(pl, tokens, k)
        G = expert_rows(BF16, a_in, layer_values[r]["W1"], pl.expert_offsets, H, 2 * I,
                        threads=threads)
        A = swiglu(G, I)
        A_in.append(a_in)
        Gs.append(G)
        As.append(A)
        values.append({"A": A, "W": layer_values[r]["W2"]})
    res = full_pipeline(w, routing, values, epoch=epoch, threads=threads)
    res.update(A_in=A_in, G=Gs, A=As)
    return res
