"""Workload definitions and seeded draws (routing, gates, operands).

The five named workloads follow the shapes of the expert-parallel down-projection
the pages describe (EpiloguePeerSink / P3PeerSendConfig: per-expert grouped GEMM
whose epilogue sends rows to the token-owning ranks; ep_signal_completion:
per-expert counts and a rank flag). The pages print no workload, so the shapes,
value laws and routing laws below are the stated synthetic recipe:

* ``tiny``             4 ranks x 2 experts, top_k 2, 64 tokens/rank, K 256 -> N 128, bf16
* ``mixtral_prefill``  8 ranks x 1 expert,  top_k 2, 4096 tokens/rank, K 14336 -> N 4096, bf16
* ``dsv3_decode``      8 ranks x 32 experts, top_k 8, 128 tokens/rank, K 2048 -> N 7168, bf16
* ``dsv3_prefill_fp8`` 8 ranks x 32 experts, top_k 8, 8192 tokens/rank, K 2048 -> N 7168,
                       e4m3 operands with 1x128 (activation) / 128x128 (weight) fp32 scales
* ``qwen3_skew``       8 ranks x 16 experts, top_k 8, 2048 tokens/rank, K 1536 -> N 4096, bf16,
                       Zipf(1.2) routing

Routing laws ("scores" per token and expert; the top_k highest are taken, slot
order = descending score, ties to the lower expert id):

* ``uniform`` iid U(0,1) scores: a uniformly random k-subset in random order.
* ``biased``  N(0,1) + per-expert bias N(0, 0.5).
* ``zipf``    log(w_e) + Gumbel noise (Plackett-Luce sampling without
              replacement). w = p^-1.2 over a seeded popularity permutation, and on
              every rank the least popular local expert gets w = 0 (so each rank
              owns an expert with no rows).

Gate laws: ``softmax_indep`` softmax of k fresh N(0,1) logits; ``softmax_sel``
softmax of the selected scores; ``sigmoid_sel`` sigmoid of the selected scores,
normalised to sum 1.

Operand laws: bf16 workloads draw A and W as N(0,1)/sqrt(K) rounded to bf16
(round to nearest even). The fp8 workload draws A and W as e4m3(N(0,1)) and the
scales as 2^U(-4,4).

Seeds: routing 1000 + id, values 2000 + id (numpy PCG64 through SeedSequence).
Large tensors are drawn in fixed 4 Mi-element chunks, chunk c seeded by
(values seed, tensor tag, rank, c), so the result does not depend on the thread
count used to draw it.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 22

_TAG_A, _TAG_W, _TAG_SA, _TAG_SW = 1, 2, 3, 4
_TAG_X, _TAG_W1 = 5, 6


@dataclass(frozen=True)
class Workload:
    name: str
    n_ranks: int
    n_local_experts: int
    top_k: int
    tokens: int  # tokens per source rank (T)
    K: int
    N: int
    dtype: str = "bf16"  # "bf16" | "fp8_1d2d"
    routing: str = "uniform"  # "uniform" | "biased" | "zipf"
    gates: str = "softmax_sel"  # "softmax_indep" | "softmax_sel" | "sigmoid_sel"
    wid: int = 0  # workload id: routing seed 1000+wid, values seed 2000+wid

    @property
    def n_experts(self) -> int:
        return self.n_ranks * self.n_local_experts

    @property
    def msg_bytes(self) -> int:
        # one bf16 output row per (token, slot)
        return 2 * self.N

    @property
    def routing_seed(self) -> int:
        return 1000 + self.wid

    @property
    def values_seed(self) -> int:
        return 2000 + self.wid


WORKLOADS = {
    "tiny": Workload("tiny", 4, 2, 2, 64, 256, 128, "bf16", "uniform", "softmax_indep", 0),
    "mixtral_prefill": Workload("mixtral_prefill", 8, 1, 2, 4096, 14336, 4096, "bf16",
                                "biased", "softmax_sel", 1),
    "dsv3_decode": Workload("dsv3_decode", 8, 32, 8, 128, 2048, 7168, "bf16",
                            "uniform", "sigmoid_sel", 2),
    "dsv3_prefill_fp8": Workload("dsv3_prefill_fp8", 8, 32, 8, 8192, 2048, 7168, "fp8_1d2d",
                                 "uniform", "sigmoid_sel", 3),
    "qwen3_skew": Workload("qwen3_skew", 8, 16, 8, 2048, 1536, 4096, "bf16",
                           "zipf", "softmax_sel", 4),
}


@dataclass
class Routing:
    topk_ids: np.ndarray  # int32 [R, T, k], global expert ids
    gates: np.ndarray  # float32 [R, T, k]
    extra: dict = field(default_factory=dict)


def _softmax(x: np.ndarray) -> np.ndarray:
    z = x - x.max(axis=-1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=-1, keepdims=True)


def make_routing(w: Workload, seed: int | None = None) -> Routing:
    """Draw top_k expert ids and gate weights for every (rank, token)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(
        w.routing_seed if seed is None else seed)))
    R, T, E, k = w.n_ranks, w.tokens, w.n_experts, w.top_k
    if k > E:
        raise ValueError("top_k larger than the expert count")
    extra = {}
    if w.routing == "uniform":
        scores = rng.random((R, T, E))
    elif w.routing == "biased":
        bias = rng.normal(0.0, 0.5, size=E)
        scores = rng.standard_normal((R, T, E)) + bias
        extra["bias"] = bias
    elif w.routing == "zipf":
        perm = rng.permutation(E)
        weight = np.empty(E)
        weight[perm] = np.arange(1, E + 1, dtype=np.float64) ** -1.2
        for r in range(R):
            local = np.arange(r * w.n_local_experts, (r + 1) * w.n_local_experts)
            weight[local[np.argmin(weight[local])]] = 0.0
        u = rng.random((R, T, E))
        gumbel = -np.log(-np.log(np.clip(u, 1e-300, 1.0 - 1e-16)))
        with np.errstate(divide="ignore"):
            scores = np.log(weight) + gumbel
        extra["weight"] = weight
    else:
        raise ValueError(f"unknown routing law {w.routing!r}")

    # descending score; a stable sort of the negated scores sends ties to the lower id
    order = np.argsort(-scores, axis=-1, kind="stable")[..., :k]
    sel = np.take_along_axis(scores, order, axis=-1)

    if w.gates == "softmax_indep":
        gates = _softmax(rng.standard_normal((R, T, k)))
    elif w.gates == "softmax_sel":
        gates = _softmax(sel)
    elif w.gates == "sigmoid_sel":
        s = 1.0 / (1.0 + np.exp(-sel))
        gates = s / s.sum(axis=-1, keepdims=True)
    else:
        raise ValueError(f"unknown gate law {w.gates!r}")
    return Routing(order.astype(np.int32), gates.astype(np.float32), extra)


def rows_per_rank(w: Workload, topk_ids: np.ndarray) -> np.ndarray:
    """Size of each rank's activation input: the number of (token, slot) entries
    routed to one of its experts (experts live on rank id // n_local_experts)."""
    return np.bincount((topk_ids.reshape(-1) // w.n_local_experts).astype(np.int64),
                       minlength=w.n_ranks)


# ----------------------------------------------------------------------------- values

def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _chunked(n: int, key: tuple, fill) -> np.ndarray:
    """Fill a flat float32 array of n draws, chunk c from SeedSequence(key + (c,))."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(c: int) -> None:
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key) + [c])))
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        fill(g, out[lo:hi])

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(min(_threads(), nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def _normal(n: int, key: tuple) -> np.ndarray:
    return _chunked(n, key, lambda g, o: g.standard_normal(out=o, dtype=np.float32))


def _log2_uniform_scale(n: int, key: tuple) -> np.ndarray:
    def fill(g, o):
        o[:] = np.exp2(g.uniform(-4.0, 4.0, size=o.shape[0])).astype(np.float32)
    return _chunked(n, key, fill)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (torch CPU)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def e4m3_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """float32 -> OCP e4m3 ("fn") bit patterns (uint8), round to nearest even (torch CPU)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def make_rank_values(w: Workload, rank: int, rows: int, seed: int | None = None) -> dict:
    """Operands of one producer rank.

    ``A`` has ``rows`` rows (the rank's routed-row count, in the receiving
    layout's row order) and ``W`` holds the rank's n_local_experts expert weights,
    [E_l, N, K] row-major (K contiguous). bf16 values are uint16 bit patterns,
    e4m3 values uint8 bit patterns.
    """
    base = w.values_seed if seed is None else seed
    K, N, El = w.K, w.N, w.n_local_experts
    out = {}
    if w.dtype == "bf16":
        s = np.float32(1.0 / np.sqrt(K))
        a = _normal(rows * K, (base, _TAG_A, rank)) * s
        out["A"] = bf16_bits_from_f32(a).reshape(rows, K)
        del a
        wt = _normal(El * N * K, (base, _TAG_W, rank)) * s
        out["W"] = bf16_bits_from_f32(wt).reshape(El, N, K)
    elif w.dtype == "fp8_1d2d":
        if K % 128 or N % 128:
            raise ValueError("blockwise fp8 needs K and N multiples of 128")
        a = _normal(rows * K, (base, _TAG_A, rank))
        out["A"] = e4m3_bits_from_f32(a).reshape(rows, K)
        del a
        wt = _normal(El * N * K, (base, _TAG_W, rank))
        out["W"] = e4m3_bits_from_f32(wt).reshape(El, N, K)
        del wt
        out["a_scales"] = _log2_uniform_scale(rows * (K // 128), (base, _TAG_SA, rank)).reshape(
            rows, K // 128)
        out["w_scales"] = _log2_uniform_scale(El * (N // 128) * (K // 128),
                                              (base, _TAG_SW, rank)).reshape(El, N // 128, K // 128)
    else:
        raise ValueError(f"unknown dtype {w.dtype!r}")
    return out


def make_layer_values(w: Workload, rank: int, seed: int | None = None) -> dict:
    """Operands of one rank for a whole MoE layer around the down-projection
    (bf16 only): the rank's tokens ``X`` [T, H] (N(0, 1)), the up/gate weights of
    its experts ``W1`` [E_l, 2I, H] (gate rows first, then up rows; N(0, 1)/sqrt(H))
    and the down-projection weights ``W2`` [E_l, H, I] (as ``make_rank_values``'s
    W). H = w.N (the hidden size the down-projection returns to), I = w.K (the
    intermediate size it reads). uint16 bf16 bit patterns."""
    if w.dtype != "bf16":
        raise ValueError("the layer operands are bf16")
    base = w.values_seed if seed is None else seed
    H, I, El = w.N, w.K, w.n_local_experts
    out = {"X": bf16_bits_from_f32(_normal(w.tokens * H, (base, _TAG_X, rank))).reshape(
        w.tokens, H)}
    out["W1"] = bf16_bits_from_f32(_normal(El * 2 * I * H, (base, _TAG_W1, rank))
                                   * np.float32(1.0 / np.sqrt(H))).reshape(El, 2 * I, H)
    out["W2"] = bf16_bits_from_f32(_normal(El * H * I, (base, _TAG_W, rank))
                                   * np.float32(1.0 / np.sqrt(I))).reshape(El, H, I)
    return out
