"""Parity of the CUDA path with the oracle, through the C ABI (GPU).

Small workloads run the oracle in full and are compared element by element:
plans, every count and flag word bit for bit; every received row and every
combined output within the tolerance; every receive slot written (the
sentinel NaN would fail the value check).
"""

import numpy as np
import pytest
import torch

import moe_expert_gemm_gb300 as ep
import oracle
from oracle.pipeline import full_pipeline
from parity_util import (TOL, assert_combine_close, assert_plan_equal, build_system,
                         make_inputs, max_rel_err, run_all)
from synth import Routing, Workload, WORKLOADS, make_routing

pytestmark = pytest.mark.gpu


def _check_full(w, routing=None, values=None, epoch=3, send_warps=-1, unfused=False,
                per_expert=False):
    routing, values = (routing, values) if values is not None else make_inputs(w, routing)
    s = build_system(w, routing, values, send_warps=send_warps, signal_mode=int(per_expert))
    run_all(s, epoch, unfused)
    torch.cuda.synchronize()
    ref = _assert_matches_oracle(s, w, routing, values, epoch, per_expert)
    return s, ref, routing, values


def _assert_matches_oracle(s, w, routing, values, epoch, per_expert=False):
    """Plans, count and flag words bit for bit; received rows and combined outputs of
    every rank within the tolerance; counters re-armed; no status bit."""
    st = s.status_words()
    assert (st == 0).all(), st
    ref = full_pipeline(w, routing, values, epoch=epoch, per_expert=per_expert)
    tol = TOL[w.dtype]
    for r in range(w.n_ranks):
        assert_plan_equal(s.plan_host(r), ref["plans"][r])
    for d in range(w.n_ranks):
        np.testing.assert_array_equal(s.counts[d].cpu().numpy().view(np.uint64), ref["counts"][d])
        got = s.recv[d].cpu().numpy().view(np.uint16)
        want = ref["recv"][d].view(np.uint16)
        assert max_rel_err(got, want) <= tol, d
        out = s.out[d].view(torch.int16).cpu().numpy().view(np.uint16)
        assert_combine_close(out, ref["out"][d], ref["out_exact"][d], ref["rows_exact"][d],
                             routing.gates[d], tol, (w.name, d))
    for r in range(w.n_ranks):  # counters re-armed for the next call
        assert int(s.atomic_counter[r].abs().sum()) == 0
        assert int(s.rank_counter[r].abs().sum()) == 0
    return ref


def test_tiny_full_parity():
    _check_full(WORKLOADS["tiny"])


def test_tiny_two_epochs_in_a_row():
    w = WORKLOADS["tiny"]
    s, ref, routing, values = _check_full(w, epoch=1)
    run_all(s, 2)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    ref2 = full_pipeline(w, routing, values, epoch=2)
    for d in range(w.n_ranks):
        np.testing.assert_array_equal(s.counts[d].cpu().numpy().view(np.uint64), ref2["counts"][d])
        out = s.out[d].view(torch.int16).cpu().numpy().view(np.uint16)
        assert_combine_close(out, ref2["out"][d], ref2["out_exact"][d], ref2["rows_exact"][d],
                             routing.gates[d], TOL[w.dtype], (w.name, "epoch 2", d))


def _fixed_routing(w, ids, seed=5):
    rng = np.random.default_rng(seed)
    g = rng.random(ids.shape).astype(np.float32) + 0.1
    return Routing(np.ascontiguousarray(ids, dtype=np.int32), (g / g.sum(-1, keepdims=True)))


EDGE = [
    # ragged tails around the 128-row tile: every token of every rank to experts 2 and 3
    ("hot_pair_ragged", Workload("hot_pair", 4, 2, 2, 100, 256, 256, "bf16", "uniform",
                                 "softmax_sel", 40), "hot"),
    ("one_row_expert", Workload("one_row", 2, 2, 1, 1, 128, 128, "bf16", "uniform",
                                "softmax_sel", 41), "random"),
    ("bm_minus_one", Workload("bm_m1", 1, 1, 1, 127, 128, 128, "bf16", "uniform",
                              "softmax_sel", 42), "random"),
    ("bm_plus_one", Workload("bm_p1", 1, 1, 1, 129, 128, 128, "bf16", "uniform",
                             "softmax_sel", 43), "random"),
    ("single_rank_topk1", Workload("r1", 1, 3, 1, 77, 192, 192, "bf16", "uniform",
                                   "softmax_sel", 44), "random"),
    ("eight_ranks_one_expert", Workload("r8", 8, 1, 2, 40, 128, 384, "bf16", "biased",
                                        "softmax_sel", 45), "random"),
    ("one_k_block", Workload("k64", 2, 2, 2, 50, 64, 128, "bf16", "uniform",
                             "softmax_sel", 46), "random"),
    ("empty_experts", Workload("empty", 4, 4, 2, 30, 256, 512, "bf16", "uniform",
                               "softmax_sel", 47), "empty"),
    ("qwen_shape_small", Workload("qwen_small", 8, 16, 8, 48, 1536, 4096, "bf16", "zipf",
                                  "softmax_sel", 48), "random"),
    # more than 32 local experts: the kernels' tile table spans several warp-wide scans
    ("many_local_experts", Workload("many_el", 2, 48, 4, 64, 128, 128, "bf16", "uniform",
                                    "softmax_sel", 73), "random"),
    ("many_local_experts_pairs", Workload("many_el_pair", 1, 40, 8, 1300, 128, 256, "bf16",
                                          "uniform", "softmax_sel", 74), "random"),
    # E_l * n_ranks above the kernels' shared-memory count cache (512 words): the
    # count words are read from the plan in global memory
    ("count_words_past_the_cache", Workload("many_counts", 8, 72, 2, 24, 128, 128, "bf16",
                                            "uniform", "softmax_sel", 79), "random"),
    # a rank whose experts receive no row at all still signals (counts 0 and its flag)
    ("rank_without_rows", Workload("idle_rank", 4, 2, 2, 40, 128, 256, "bf16", "uniform",
                                   "softmax_sel", 80), "idle_rank"),
    # a top_k with no specialised combine (3)
    ("topk3", Workload("topk3", 4, 2, 3, 40, 128, 256, "bf16", "uniform", "softmax_sel", 55),
     "random"),
    # blockwise fp8: several scale blocks along K and N, ragged tails, empty experts
    ("fp8_small", Workload("fp8_small", 4, 4, 2, 100, 384, 512, "fp8_1d2d", "uniform",
                           "sigmoid_sel", 51), "random"),
    ("fp8_zipf_empty", Workload("fp8_zipf", 4, 4, 4, 90, 256, 256, "fp8_1d2d", "zipf",
                                "sigmoid_sel", 52), "random"),
    ("fp8_dsv3_shape_small", Workload("fp8_dsv3_small", 8, 32, 8, 64, 2048, 7168, "fp8_1d2d",
                                      "uniform", "sigmoid_sel", 53), "random"),
    # N % 256 = 128: the fp8 kernel's 128-column tiles (four partial buffers)
    ("fp8_128_column_tiles", Workload("fp8_n384", 4, 2, 2, 80, 384, 384, "fp8_1d2d", "uniform",
                                      "sigmoid_sel", 77), "random"),
]


_EDGE = {name: w for name, w, _ in EDGE}  # edge workloads by name


@pytest.mark.parametrize("name,w,kind", EDGE, ids=[e[0] for e in EDGE])
def test_edge_parity(name, w, kind):
    routing = make_routing(w)
    if kind == "hot":
        ids = np.tile(np.array([2, 3], np.int32), (w.n_ranks, w.tokens, 1))
        routing = _fixed_routing(w, ids)
    elif kind == "idle_rank":
        # experts 2 and 3 (rank 1's) receive nothing
        rng = np.random.default_rng(11)
        choices = np.array([0, 1, 4, 5, 6, 7], np.int32)
        ids = np.stack([np.stack([rng.choice(choices, w.top_k, replace=False)
                                  for _ in range(w.tokens)]) for _ in range(w.n_ranks)])
        routing = _fixed_routing(w, ids)
    elif kind == "empty":
        # only experts 0, 5, 6 and 13 receive rows; every rank keeps at least one empty expert
        rng = np.random.default_rng(9)
        choices = np.array([0, 5, 6, 13], np.int32)
        ids = np.stack([np.stack([rng.choice(choices, 2, replace=False) for _ in range(w.tokens)])
                        for _ in range(w.n_ranks)])
        routing = _fixed_routing(w, ids)
    _check_full(w, routing)


@pytest.mark.parametrize("T", [200, 1100])  # single CTAs / CTA pairs (T*top_k/E_l >= 256)
def test_identity_weights_bit_exact(T):
    """W_e = 2^c I, top_k = 1, gate 1: the whole path moves the activation rows,
    scaled by a power of two, bit for bit."""
    w = Workload("ident_gpu", 4, 2, 1, T, 256, 256, "bf16", "uniform", "softmax_indep", 49)
    routing, values = make_inputs(w)
    routing.gates[:] = 1.0
    for q in range(w.n_ranks):
        eye = np.stack([np.eye(w.N, dtype=np.float32) * 2.0 ** (e - q)
                        for e in range(w.n_local_experts)])
        values[q]["W"] = torch.from_numpy(eye).to(torch.bfloat16).view(torch.int16).numpy().view(
            np.uint16)
    s = build_system(w, routing, values)
    run_all(s, 1)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    ref = full_pipeline(w, routing, values, epoch=1)
    for d in range(w.n_ranks):
        np.testing.assert_array_equal(s.recv[d].cpu().numpy(), ref["recv"][d])
        np.testing.assert_array_equal(s.out[d].view(torch.int16).cpu().numpy().view(np.uint16),
                                      ref["out"][d])


@pytest.mark.parametrize("send_warps", [-1, 4])
def test_local_store_when_sink_disabled(send_warps):
    """p3_control < 0: rows go to the local C in plan order, nothing is sent or signalled."""
    w = WORKLOADS["tiny"]
    routing, values = make_inputs(w)
    s = build_system(w, routing, values, send_warps=send_warps)
    r = 1
    m = s.plan_host(r)["m_total"]
    C = torch.zeros((s.ops[r]["A"].shape[0], w.N), dtype=torch.bfloat16, device="cuda")
    s.send(r, epoch=7, p3_control=-1, C=C)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    for d in range(w.n_ranks):  # untouched
        assert (s.recv[d].cpu().numpy() == 0xFF).all()
        assert (s.counts[d].cpu().numpy() == -1).all()
    pl = oracle.plan(w.n_ranks, w.n_local_experts, w.top_k, routing.topk_ids, r)
    Y = oracle.expert_rows(oracle.BF16, values[r]["A"], values[r]["W"], pl.expert_offsets, w.K,
                           w.N)
    got = C[:m].view(torch.int16).cpu().numpy().view(np.uint16)
    assert max_rel_err(got, Y) <= TOL["bf16"]


@pytest.mark.parametrize("N,T,pair,send_warps", [(384, 300, False, -1), (512, 600, True, -1),
                                                 (512, 600, True, 4), (384, 300, False, 4)])
def test_trace_records_every_tile_once(N, T, pair, send_warps):
    """Optional per-tile timestamps: every tile appears once per CTA that works on
    it (single CTAs: once; 256-column bf16 tiles on CTA pairs: once per CTA of the
    pair), times are ordered, and exactly the non-empty experts are marked as
    completed, once each. With dedicated send warps the stored time is taken by
    the send warps, after the output warps have handed over every sub-tile."""
    w = Workload("trace_small", 4, 4, 2, T, 256, N, "bf16", "zipf", "softmax_sel", 50)
    routing, values = make_inputs(w)
    s = build_system(w, routing, values, send_warps=send_warps)
    for r in range(w.n_ranks):
        s.send(r, epoch=1)
    tr = s.send_traced(1, epoch=2, records=64)
    assert (s.status_words() == 0).all()
    recs = [rec for b in tr for rec in b["records"]]
    assert sum(b["tiles"] for b in tr) == len(recs)
    pl = oracle.plan(w.n_ranks, w.n_local_experts, w.top_k, routing.topk_ids, 1)
    rows = np.diff(pl.expert_offsets)
    bn = 256 if N % 256 == 0 else (128 if N % 128 == 0 else 64)  # widest column block
    tile_rows, n_blocks, copies = (256, N // bn, 2) if pair else (128, N // bn, 1)
    n_tiles = int((-(-rows // tile_rows)).sum()) * n_blocks
    assert sorted(r["tile"] for r in recs) == sorted(list(range(n_tiles)) * copies)
    assert all(b["t_start"] <= r["t_ready"] <= r["t_stored"] <= r["t_done"]
               for b in tr for r in b["records"])
    done = sorted(r["expert"] for r in recs if r["completed"])
    assert done == [e for e in range(w.n_local_experts) if rows[e] > 0]


def test_maximum_local_experts_parity():
    """EP_MAX_LOCAL_EXPERTS (256) local experts in one fused call: a tile table over
    256 experts (most with one to three rows, many empty) and E_l * R count words."""
    w = Workload("max_el", 2, ep.EP_MAX_LOCAL_EXPERTS, 8, 64, 128, 128, "bf16", "uniform",
                 "softmax_sel", 94)
    _check_full(w)


@pytest.mark.parametrize("signal_mode", [0, 1])
def test_empty_batch_signals_every_expert_with_count_zero(signal_mode):
    """A batch with no tokens (receive buffers sized for 16): every expert of every
    rank still signals ("ep_signal_completion": an empty (expert, destination) segment
    reports count 0, and the rank flag needs every expert), the combine has nothing to
    reduce, and no receive slot is written."""
    from moe_expert_gemm_gb300.system import EpSystem
    R, El, k, K, N = 4, 2, 2, 128, 128
    s = EpSystem(R, El, k, 0, K, N, "bf16", max_tokens=16, signal_mode=signal_mode)
    s.set_routing(np.zeros((R, 0, k), np.int32))
    for r in range(R):
        s.plan(r)
        s.set_operands(r, np.zeros((0, K), np.uint16), np.zeros((El, N, K), np.uint16))
        s.set_gates(r, np.zeros((0, k), np.float32))
    for r in range(R):
        s.send(r, epoch=7)
    for d in range(R):
        s.combine(d, epoch=7)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all(), s.status_words()
    for d in range(R):
        words = s.counts[d].cpu().numpy().view(np.uint64)
        if signal_mode == 0:
            np.testing.assert_array_equal(words[:El * R], np.zeros(El * R, np.uint64))
            np.testing.assert_array_equal(words[El * R:], np.full(R, 7, np.uint64))
        else:
            np.testing.assert_array_equal(words[:El * R], np.full(El * R, 7 << 32, np.uint64))
        assert (s.recv[d].cpu().numpy() == 0xFF).all()  # the sentinel everywhere
    for r in range(R):
        assert s.plan_host(r)["m_total"] == 0
        assert int(s.atomic_counter[r].abs().sum()) == 0
        assert int(s.rank_counter[r].abs().sum()) == 0


def test_pair_kernel_small_parity():
    """256-column bf16 tiles run on CTA pairs (M = 256 across two SMs) once an
    expert's expected rows fill a pair tile: ragged experts that end inside
    either CTA's half of a pair tile, empty experts."""
    w = Workload("pair_small", 4, 3, 2, 400, 320, 512, "bf16", "zipf", "softmax_sel", 54)
    _check_full(w)


def test_fp8_many_rows_per_expert_parity():
    """Blockwise fp8 with several 128-row blocks per expert: ragged experts, several
    scale blocks along K and N."""
    w = Workload("fp8_pair_small", 2, 2, 2, 400, 384, 512, "fp8_1d2d", "zipf", "sigmoid_sel", 56)
    _check_full(w)


SEND_WARP_CASES = [
    # 256-, 128- and 64-column tiles; ragged tails; empty experts; eight ranks; a
    # shape that would otherwise run on CTA pairs
    ("tiny", WORKLOADS["tiny"]),
    ("bn256_ragged", Workload("sw256", 4, 2, 2, 100, 256, 256, "bf16", "uniform",
                              "softmax_sel", 60)),
    ("bn128_eight_ranks", Workload("sw128", 8, 1, 2, 40, 128, 384, "bf16", "biased",
                                   "softmax_sel", 61)),
    ("bn64_single_rank", Workload("sw64", 1, 3, 1, 77, 192, 192, "bf16", "uniform",
                                  "softmax_sel", 62)),
    ("pair_shape", Workload("sw_pair", 4, 3, 2, 400, 320, 512, "bf16", "zipf",
                            "softmax_sel", 63)),
    ("qwen_shape_small", Workload("sw_qwen", 8, 16, 8, 48, 1536, 4096, "bf16", "zipf",
                                  "softmax_sel", 64)),
    # CTA pairs with send warps: several pair tiles per pair, ragged row blocks
    ("pair_many_tiles", Workload("sw_pair_many", 8, 2, 2, 1000, 512, 1024, "bf16", "biased",
                                 "softmax_sel", 66)),
]


@pytest.mark.parametrize("name,w", SEND_WARP_CASES, ids=[c[0] for c in SEND_WARP_CASES])
def test_dedicated_send_warps_parity(name, w):
    """send_warps = 4: four send warps, one per output warp, store the rows the
    output warps stage in two slots each. Same plans, counts, flags, rows and
    combined outputs as the inline sink; counters re-armed."""
    _check_full(w, send_warps=4)


def test_dedicated_send_warps_two_epochs_and_empty_experts():
    w = Workload("sw_empty", 4, 4, 2, 30, 256, 512, "bf16", "uniform", "softmax_sel", 65)
    rng = np.random.default_rng(10)
    choices = np.array([0, 5, 6, 13], np.int32)
    ids = np.stack([np.stack([rng.choice(choices, 2, replace=False) for _ in range(w.tokens)])
                    for _ in range(w.n_ranks)])
    routing = _fixed_routing(w, ids)
    s, ref, routing, values = _check_full(w, routing, epoch=5, send_warps=4)
    run_all(s, 6)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    ref2 = full_pipeline(w, routing, values, epoch=6)
    for d in range(w.n_ranks):
        np.testing.assert_array_equal(s.counts[d].cpu().numpy().view(np.uint64), ref2["counts"][d])


FP8_ROW_BLOCK_CASES = [
    # several 128-row blocks per expert with ragged last blocks; zipf routing leaves
    # experts empty; 256- and 128-column tiles; one K block; eight ranks
    ("bn256_zipf_empty", Workload("fp8_rb_zipf", 4, 4, 4, 300, 256, 768, "fp8_1d2d", "zipf",
                                  "sigmoid_sel", 57)),
    ("bn128_ragged", Workload("fp8_rb_128", 2, 2, 2, 300, 256, 384, "fp8_1d2d", "uniform",
                              "sigmoid_sel", 58)),
    ("pair_one_k_block", Workload("fp8_p1k", 2, 3, 2, 500, 128, 256, "fp8_1d2d", "uniform",
                                  "sigmoid_sel", 84)),
    ("pair_eight_ranks", Workload("fp8_p8", 8, 4, 4, 300, 256, 384, "fp8_1d2d", "biased",
                                  "sigmoid_sel", 85)),
]


@pytest.mark.parametrize("name,w", FP8_ROW_BLOCK_CASES, ids=[c[0] for c in FP8_ROW_BLOCK_CASES])
def test_fp8_row_block_parity(name, w):
    _check_full(w)


def test_fp8_many_rows_per_expert_signal_modes():
    """Blockwise fp8 with several row blocks per expert under per-expert signals, and
    with the sink disabled (rows to a local C, then ep_scatter_send)."""
    w = Workload("fp8_modes", 4, 2, 2, 400, 256, 512, "fp8_1d2d", "zipf", "sigmoid_sel", 86)
    _check_full(w, per_expert=True)
    _check_full(w, unfused=True)


@pytest.mark.parametrize("T", [100, 600])  # one / several row blocks per expert
def test_fp8_identity_weights_bit_exact(T):
    """Blockwise fp8 with W_e = I (e4m3 1.0 on the diagonal), power-of-two scales,
    top_k = 1, gate 1: y[m, n] = sa[m, n/128] * sw[e, n/128, n/128] * a8[m, n] is
    exact in bf16, so rows and combined outputs match the oracle bit for bit."""
    w = Workload("ident_fp8", 4, 2, 1, T, 256, 256, "fp8_1d2d", "uniform", "softmax_indep", 59)
    routing, values = make_inputs(w)
    routing.gates[:] = 1.0
    rng = np.random.default_rng(11)
    for q in range(w.n_ranks):
        v = values[q]
        v["W"] = np.zeros_like(v["W"])
        for e in range(w.n_local_experts):
            np.fill_diagonal(v["W"][e], 0x38)  # e4m3 1.0
        v["a_scales"] = np.exp2(rng.integers(-4, 5, v["a_scales"].shape)).astype(np.float32)
        v["w_scales"] = np.exp2(rng.integers(-4, 5, v["w_scales"].shape)).astype(np.float32)
    s = build_system(w, routing, values)
    run_all(s, 1)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    ref = full_pipeline(w, routing, values, epoch=1)
    for d in range(w.n_ranks):
        np.testing.assert_array_equal(s.recv[d].cpu().numpy(), ref["recv"][d])
        np.testing.assert_array_equal(s.out[d].view(torch.int16).cpu().numpy().view(np.uint16),
                                      ref["out"][d])


UNFUSED_CASES = [
    ("tiny", WORKLOADS["tiny"]),
    ("hot_pair_ragged", _EDGE["hot_pair_ragged"]),
    ("eight_ranks_one_expert", _EDGE["eight_ranks_one_expert"]),
    ("pair_shape", Workload("uf_pair", 4, 3, 2, 400, 320, 512, "bf16", "zipf", "softmax_sel", 66)),
    ("fp8_small", _EDGE["fp8_small"]),
]


@pytest.mark.parametrize("name,w", UNFUSED_CASES, ids=[c[0] for c in UNFUSED_CASES])
def test_unfused_send_parity(name, w):
    """The unfused comparator (sink disabled: rows to a local C; then
    ep_scatter_send) delivers the same rows, counts and flags as the fused call."""
    routing, values = make_inputs(w)
    if name == "hot_pair_ragged":
        ids = np.tile(np.array([2, 3], np.int32), (w.n_ranks, w.tokens, 1))
        routing = _fixed_routing(w, ids)
    s, ref, routing, values = _check_full(w, routing, epoch=4, unfused=True)
    # a second call re-arms the block counter and publishes the new epoch
    run_all(s, 5, unfused=True)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    for d in range(w.n_ranks):
        flags = s.counts[d].cpu().numpy().view(np.uint64)[w.n_local_experts * w.n_ranks:]
        assert (flags == 5).all()
        assert int(s.block_counter[d].item()) == 0


PER_EXPERT_CASES = [
    ("tiny", WORKLOADS["tiny"], False),
    ("empty_experts", _EDGE["empty_experts"], False),
    ("eight_ranks_one_expert", _EDGE["eight_ranks_one_expert"], False),
    ("topk3", _EDGE["topk3"], False),
    ("pair_shape", Workload("pe_pair", 4, 3, 2, 400, 320, 512, "bf16", "zipf", "softmax_sel", 67),
     False),
    ("fp8_small", _EDGE["fp8_small"], False),
    ("many_local_experts", _EDGE["many_local_experts"], False),
    ("count_words_past_the_cache", _EDGE["count_words_past_the_cache"], False),
    ("tiny_unfused", WORKLOADS["tiny"], True),
]


@pytest.mark.parametrize("name,w,unfused", PER_EXPERT_CASES, ids=[c[0] for c in PER_EXPERT_CASES])
def test_per_expert_signalling_parity(name, w, unfused):
    """EP_SIGNAL_PER_EXPERT (the pages' default mode): every expert's count word is an
    epoch-tagged arrival signal, no rank flag is written, and the combine waits per
    token for that token's experts. Same rows and outputs; count words as the oracle's
    per-expert signalling writes them (flag words untouched)."""
    routing = None
    if name == "empty_experts":
        rng = np.random.default_rng(9)
        choices = np.array([0, 5, 6, 13], np.int32)
        ids = np.stack([np.stack([rng.choice(choices, 2, replace=False) for _ in range(w.tokens)])
                        for _ in range(w.n_ranks)])
        routing = _fixed_routing(w, ids)
    _check_full(w, routing, epoch=2**32 + 9, unfused=unfused, per_expert=True)


def test_per_expert_tokens_of_finished_ranks_are_combined_while_one_rank_is_missing():
    """With per-expert signals a token is reduced once its own experts have arrived:
    when rank 3 never sends, exactly the tokens routed to one of rank 3's experts
    time out (left unwritten, EP_STATUS_TIMEOUT); every other token is combined."""
    w = WORKLOADS["tiny"]
    routing, values = make_inputs(w)
    s = build_system(w, routing, values, timeout_ns=30_000_000, signal_mode=1)
    for r in range(w.n_ranks):
        if r != 3:
            s.send(r, epoch=1)
    for d in range(w.n_ranks):
        s.out[d].fill_(0)
        s.combine(d, epoch=1)
    torch.cuda.synchronize()
    assert s.status_words()[2] & ep.EP_STATUS_TIMEOUT
    ref = full_pipeline(w, routing, values, epoch=1, per_expert=True)
    missing = routing.topk_ids // w.n_local_experts == 3
    for d in range(w.n_ranks):
        out = s.out[d].view(torch.int16).cpu().numpy().view(np.uint16)
        waits = missing[d].any(axis=1)
        assert waits.any() and (~waits).any()
        assert (out[waits] == 0).all()
        assert_combine_close(out[~waits], ref["out"][d][~waits], ref["out_exact"][d][~waits],
                             ref["rows_exact"][d][~waits], routing.gates[d][~waits], TOL["bf16"],
                             (w.name, "missing rank", d))


OVERLAP_CASES = [
    ("tiny", WORKLOADS["tiny"], 0),
    ("qwen_shape_small", _EDGE["qwen_shape_small"], 0),
    ("pair_shape", Workload("ov_pair", 4, 3, 2, 400, 320, 512, "bf16", "zipf", "softmax_sel", 68),
     0),
    ("fp8_small", _EDGE["fp8_small"], 0),
    ("tiny_per_expert", WORKLOADS["tiny"], 1),
]


@pytest.mark.parametrize("name,w,signal_mode", OVERLAP_CASES, ids=[c[0] for c in OVERLAP_CASES])
def test_combine_overlapping_the_fused_send(name, w, signal_mode):
    """The combine launched as a programmatic dependent of the destination's own
    fused send (the last producer to run) starts before that send has ended; its
    rows are ordered by the flags (or count words) it acquires, so the outputs
    still match the oracle."""
    routing, values = make_inputs(w)
    s = build_system(w, routing, values, signal_mode=signal_mode)
    for d in range(w.n_ranks):
        for r in range(w.n_ranks):
            if r != d:
                s.send(r, epoch=10 + d)
        s.send(d, epoch=10 + d)  # d's own send, then its combine right behind it
        s.combine(d, epoch=10 + d, overlap=ep.EP_OVERLAP_INPUTS_READY)
        torch.cuda.synchronize()
        assert (s.status_words() == 0).all(), (d, s.status_words())
        ref = full_pipeline(w, routing, values, epoch=10 + d, per_expert=bool(signal_mode))
        out = s.out[d].view(torch.int16).cpu().numpy().view(np.uint16)
        assert_combine_close(out, ref["out"][d], ref["out_exact"][d], ref["rows_exact"][d],
                             routing.gates[d], TOL[w.dtype], (w.name, "overlap", d))


SEND_OVERLAP_CASES = [
    ("tiny", WORKLOADS["tiny"]),
    ("qwen_shape_small", _EDGE["qwen_shape_small"]),
    ("pair_shape", Workload("so_pair", 4, 3, 2, 400, 320, 512, "bf16", "zipf", "softmax_sel", 78)),
    ("fp8_small", _EDGE["fp8_small"]),
]


@pytest.mark.parametrize("name,w", SEND_OVERLAP_CASES, ids=[c[0] for c in SEND_OVERLAP_CASES])
def test_send_overlapping_the_plan_that_feeds_it(name, w):
    """Each rank's plan is recomputed into fresh buffers by the kernel right before an
    overlapped send (a programmatic dependent of it), and each combine overlaps the
    send before it: the send must read the plan only after the plan kernel's memory
    is visible, and the results must be the oracle's."""
    routing, values = make_inputs(w)
    s = build_system(w, routing, values)
    torch.cuda.synchronize()
    epoch = 4
    for r in range(w.n_ranks):
        s.plan(r)
        s.send(r, epoch, overlap=True)
    for d in range(w.n_ranks):
        s.combine(d, epoch, overlap=ep.EP_OVERLAP_INPUTS_READY)
    torch.cuda.synchronize()
    _assert_matches_oracle(s, w, routing, values, epoch)


def test_combine_overlapping_the_kernel_that_writes_its_gates():
    """The combine launched as a programmatic dependent of a kernel that writes its
    gates (an elementwise kernel right before it) reads the new gates: it waits for
    that kernel's completion before reading them."""
    w = WORKLOADS["tiny"]
    routing, values = make_inputs(w)
    s = build_system(w, routing, values)
    run_all(s, 1)
    torch.cuda.synchronize()
    rng = np.random.default_rng(21)
    g2 = rng.random(routing.gates.shape).astype(np.float32) + 0.1
    g2 /= g2.sum(-1, keepdims=True)
    g2_dev = torch.from_numpy(g2).cuda()
    for d in range(w.n_ranks):
        torch.mul(g2_dev[d], 1.0, out=s.gates[d])  # a kernel, right before the combine
        s.combine(d, epoch=1, overlap=ep.EP_OVERLAP_ANY)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    ref = full_pipeline(w, Routing(routing.topk_ids, g2), values, epoch=1)
    for d in range(w.n_ranks):
        out = s.out[d].view(torch.int16).cpu().numpy().view(np.uint16)
        assert_combine_close(out, ref["out"][d], ref["out_exact"][d], ref["rows_exact"][d], g2[d],
                             TOL["bf16"], (w.name, "gate writer", d))
