"""Parity at the full workload sizes, in the launch configuration the benchmark
times (every producer rank once, then rank 0's combine), checked where the
oracle can afford it: every plan, count and flag word bit for bit; every receive
slot of rank 0 written; sampled received rows and combined outputs of rank 0
and sampled rows rank 0 sent to the other ranks within the tolerance."""

import numpy as np
import pytest
import torch

import oracle
from oracle.pipeline import SENTINEL_WORD, sampled_pipeline
from parity_util import (TOL, assert_combine_close, assert_plan_equal, build_system,
                         make_inputs, max_rel_err)
from synth import WORKLOADS, Workload

pytestmark = pytest.mark.gpu


MEDIUM = {
    # many rows per expert and wide W blocks: the kernel walks row blocks fastest
    "fp8_rows_fastest": Workload("fp8_rows_fastest", 2, 2, 2, 4096, 256, 7168, "fp8_1d2d",
                                 "uniform", "sigmoid_sel", 60),
}


CASES = [(n, "fused", 0) for n in ("mixtral_prefill", "dsv3_decode", "qwen3_skew",
                                   "dsv3_prefill_fp8", "fp8_rows_fastest")] + [
    # the other producer and signalling forms at full size
    ("qwen3_skew", "unfused", 0), ("dsv3_decode", "fused", 1), ("mixtral_prefill", "unfused", 1),
    ("dsv3_prefill_fp8", "fused", 1)]


@pytest.mark.parametrize("name,path,signal_mode", CASES,
                         ids=[f"{n}-{p}-{'per_expert' if m else 'rank_flag'}"
                              for n, p, m in CASES])
def test_full_size_sampled_parity(name, path, signal_mode):
    w = WORKLOADS[name] if name in WORKLOADS else MEDIUM[name]
    R, El, k, T, N = w.n_ranks, w.n_local_experts, w.top_k, w.tokens, w.N
    routing, values = make_inputs(w)
    s = build_system(w, routing, values, signal_mode=signal_mode)
    for r in range(R):
        if path == "unfused":
            s.send_unfused(r, 1, s.local_C(r))
        else:
            s.send(r, epoch=1)
    s.combine(0, epoch=1)
    torch.cuda.synchronize()
    st = s.status_words()
    assert (st == 0).all(), st

    plans = {r: oracle.plan(R, El, k, routing.topk_ids, r) for r in range(R)}
    for r in range(R):
        assert_plan_equal(s.plan_host(r), plans[r])
    counts = [np.full(El * R + R, SENTINEL_WORD, np.uint64) for _ in range(R)]
    for r in range(R):
        if signal_mode:
            oracle.signal_per_expert(R, El, r, plans[r].send_counts, 1, counts)
        else:
            oracle.signal(R, El, r, plans[r].send_counts, 1, counts, np.zeros(R, np.int32))
    for d in range(R):
        np.testing.assert_array_equal(s.counts[d].cpu().numpy().view(np.uint64), counts[d])

    recv0 = s.recv[0].cpu().numpy().view(np.uint16).reshape(T, k, N)
    assert not (recv0 == 0xFFFF).any(), "a receive slot of rank 0 was never written"

    rng = np.random.default_rng(17)
    toks = np.sort(rng.choice(T, size=min(T, 48), replace=False))
    ref = sampled_pipeline(w, routing, lambda r: values[r], 0, toks, plans=plans)
    tol = TOL[w.dtype]
    assert max_rel_err(recv0[toks], ref["rows"]) <= tol
    out0 = s.out[0].view(torch.int16).cpu().numpy().view(np.uint16)
    assert_combine_close(out0[toks], ref["out"], ref["out_exact"], ref["rows_exact"],
                         routing.gates[0][toks], tol, (w.name, "sampled", 0))

    # rows rank 0 produced for the other ranks
    p0 = plans[0]
    ms = np.sort(rng.choice(p0.m_total, size=min(p0.m_total, 32), replace=False))
    v0 = values[0]
    Y = oracle.expert_rows(oracle.BF16 if w.dtype == "bf16" else oracle.FP8_1D2D, v0["A"],
                           v0["W"], p0.expert_offsets, w.K, N, rows=ms,
                           a_scales=v0.get("a_scales"), w_scales=v0.get("w_scales"))
    bufs = {}
    for i, m in enumerate(ms):
        e = int(np.searchsorted(p0.expert_offsets, m, side="right") - 1)
        dst = int(np.searchsorted(p0.seg_offsets[e], m, side="right") - 1)
        t, j = p0.src_info[m]
        if dst not in bufs:
            bufs[dst] = s.recv[dst].cpu().numpy().view(np.uint16).reshape(T, k, N)
        assert max_rel_err(bufs[dst][t, j], Y[i]) <= tol, (m, dst, t, j)
