"""Pins of the oracle to things other than itself (no GPU needed).

Each test checks one oracle function against a library routine, a closed form,
a hand-worked value from the pages' formulas, brute force on tiny inputs, or a
special case with an exact answer, so that a dropped term, a wrong index, a
swapped operand or a double rounding in the oracle fails at least one of them.
"""

import os

import numpy as np
import pytest
import torch

import oracle
from oracle.pipeline import full_pipeline, sampled_pipeline
from synth import Workload, WORKLOADS, make_rank_values, make_routing, rows_per_rank

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# ----------------------------------------------------------------- formats


def _torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_matches_torch_on_binary32_values():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # force exact ties (low half = 0x8000) on a quarter of them, both parities
    bits[::4] = (bits[::4] & 0xFFFF0000) | 0x8000
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    extra = np.array([0.0, -0.0, 1e-45, -1e-45, 1.1754944e-38, 3.3895e38, 3.3896e38, 3.4e38,
                      -3.4e38, 1.0, 1.00390625, 1.01171875], dtype=np.float32)
    x = np.concatenate([x, extra])
    got = oracle.bf16_from_f64(x.astype(np.float64))
    want = _torch_bf16_bits(x)
    np.testing.assert_array_equal(got, want)


def test_bf16_rne_rounds_doubles_once():
    # closed forms: 1 + 2^-8 is the midpoint of 1.0 and 1 + 2^-7
    cases = {
        1 + 2.0**-8: 0x3F80,                  # tie -> even (1.0)
        1 + 3 * 2.0**-8: 0x3F82,              # tie between 0x3F81 and 0x3F82 -> even
        1 + 2.0**-8 + 2.0**-40: 0x3F81,       # just above the midpoint
        1 + 2.0**-8 + 2.0**-30: 0x3F81,       # binary32 would round to the midpoint first
        -(1 + 2.0**-8 + 2.0**-30): 0xBF81,
        2.0**-133: 0x0001,                    # smallest bf16 subnormal
        2.0**-134: 0x0000,                    # half of it: tie -> even (zero)
        3 * 2.0**-135: 0x0001,
        2.0**128: 0x7F80,
        (2 - 2.0**-7) * 2.0**127: 0x7F7F,     # largest finite
        (2 - 2.0**-8) * 2.0**127: 0x7F80,     # midpoint above it rounds (to even) to inf
    }
    for x, bits in cases.items():
        assert int(oracle.bf16_from_f64(np.array([x]))[0]) == bits, (x, hex(bits))


def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f64(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_f64(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert nan.sum() == 2  # S.1111.111
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0**-9


# ---------------------------------------------------------- index formulas


def test_index_formulas_golden():
    n = 0
    with open(os.path.join(GOLDEN, "index_formulas.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            kind, *vals = line
            vals = list(map(int, vals))
            if kind == "recv_count":
                e, rk, R, want = vals
                assert oracle.recv_count_index(e, rk, R) == want
            else:
                s, j, b, k, msg, want = vals
                assert oracle.recv_buf_offset(s, j, b, k, msg) == want
            n += 1
    assert n >= 10


@pytest.mark.parametrize("T,k,N", [(5, 3, 8), (64, 2, 128), (3, 8, 64)])
def test_recv_buf_layout_is_a_bijection(T, k, N):
    msg = 2 * N
    offs = sorted(oracle.recv_buf_offset(t, j, 2 * n, k, msg)
                  for t in range(T) for j in range(k) for n in range(N))
    assert offs == list(range(0, T * k * msg, 2))


def test_recv_count_layout_is_a_bijection():
    for El, R in [(1, 8), (2, 4), (32, 8), (16, 8)]:
        idx = sorted(oracle.recv_count_index(e, rk, R) for e in range(El) for rk in range(R))
        assert idx == list(range(El * R))


# -------------------------------------------------------------------- plan


def _brute_plan(topk, R, El, rank):
    """Row order from a sort of (local expert, source rank, token, slot) keys."""
    keys = []
    Rr, T, k = topk.shape
    for rk in range(Rr):
        for t in range(T):
            for j in range(k):
                g = int(topk[rk, t, j])
                if g // El == rank:
                    keys.append((g % El, rk, t, j))
    keys.sort()
    return keys



def _edge_routings():
    rng = np.random.default_rng(3)
    out = []
    # every token of every rank to the same two experts of rank 1 (other experts empty)
    R, El, k, T = 4, 2, 2, 9
    out.append((R, El, k, np.tile(np.array([2, 3], np.int32), (R, T, 1))))
    # top_k = 1, single rank
    out.append((1, 3, 1, rng.integers(0, 3, size=(1, 17, 1)).astype(np.int32)))
    # 8 ranks, one expert each, top_k = 2 distinct
    ids = np.stack([np.stack([rng.choice(8, 2, replace=False) for _ in range(33)])
                    for _ in range(8)]).astype(np.int32)
    out.append((8, 1, 2, ids))
    return out


@pytest.mark.parametrize("case", range(4))
def test_plan_matches_brute_force(case):
    if case == 0:
        w = WORKLOADS["tiny"]
        R, El, k, ids = w.n_ranks, w.n_local_experts, w.top_k, make_routing(w).topk_ids
    else:
        R, El, k, ids = _edge_routings()[case - 1]
    T = ids.shape[1]
    for rank in range(R):
        pl = oracle.plan(R, El, k, ids, rank)
        keys = _brute_plan(ids, R, El, rank)
        assert pl.m_total == len(keys)
        np.testing.assert_array_equal(pl.src_info, np.array([(t, j) for _, _, t, j in keys],
                                                            np.int32).reshape(-1, 2))
        np.testing.assert_array_equal(
            pl.gather_idx, np.array([(rk * T + t) * k + j for _, rk, t, j in keys], np.int32))
        for e in range(El):
            rows_e = [i for i, key in enumerate(keys) if key[0] == e]
            start = rows_e[0] if rows_e else sum(1 for key in keys if key[0] < e)
            assert pl.expert_offsets[e] == start
            for rk in range(R):
                cnt = sum(1 for key in keys if key[0] == e and key[1] == rk)
                assert pl.send_counts[e, rk] == cnt
                assert pl.seg_offsets[e, rk] == sum(
                    1 for key in keys if (key[0], key[1]) < (e, rk))
        assert pl.expert_offsets[El] == len(keys)


def test_plan_counts_cover_every_token_slot():
    w = WORKLOADS["tiny"]
    ids = make_routing(w).topk_ids
    R, El, k, T = w.n_ranks, w.n_local_experts, w.top_k, w.tokens
    per_dst = np.zeros(R, np.int64)
    for r in range(R):
        per_dst += oracle.plan(R, El, k, ids, r).send_counts.sum(axis=0)
    np.testing.assert_array_equal(per_dst, np.full(R, T * k))
    np.testing.assert_array_equal(rows_per_rank(w, ids),
                                  [oracle.plan(R, El, k, ids, r).m_total for r in range(R)])


def test_plan_rejects_bad_ids_and_capacity():
    ids = np.zeros((2, 3, 1), np.int32)
    ids[1, 2, 0] = 4  # experts 0..3 exist
    with pytest.raises(ValueError):
        oracle.plan(2, 2, 1, ids, 0)
    with pytest.raises(ValueError):
        oracle.plan(2, 2, 1, np.zeros((2, 3, 1), np.int32), 0, max_rows=5)


# ------------------------------------------------------------- expert rows


def _ulp_ok(got_bits, ref, rel=2.0**-8):
    """Correct rounding of ref to 8 significant bits has relative error <= 2^-9;
    allow one more binade of slack for summation-order differences."""
    got = oracle.bf16_to_f64(got_bits)
    tiny = 2.0**-120
    return np.all(np.abs(got - ref) <= rel * np.abs(ref) + tiny)


def test_expert_rows_bf16_matches_numpy_matmul():
    w = WORKLOADS["tiny"]
    r = make_routing(w)
    m = int(rows_per_rank(w, r.topk_ids)[1])
    v = make_rank_values(w, 1, m)
    pl = oracle.plan(w.n_ranks, w.n_local_experts, w.top_k, r.topk_ids, 1)
    Y = oracle.expert_rows(oracle.BF16, v["A"], v["W"], pl.expert_offsets, w.K, w.N)
    A = torch.from_numpy(v["A"].view(np.int16)).view(torch.bfloat16).double().numpy()
    W = torch.from_numpy(v["W"].view(np.int16)).view(torch.bfloat16).double().numpy()
    for e in range(w.n_local_experts):
        lo, hi = pl.expert_offsets[e], pl.expert_offsets[e + 1]
        ref = A[lo:hi] @ W[e].T
        assert _ulp_ok(Y[lo:hi], ref)
        # a transposed or wrong-expert weight is far off
        other = A[lo:hi] @ W[1 - e].T
        assert not _ulp_ok(Y[lo:hi], other)


def test_unrounded_rows_and_exact_combine_match_numpy():
    w = WORKLOADS["tiny"]
    r = make_routing(w)
    m = rows_per_rank(w, r.topk_ids)
    vals = [make_rank_values(w, q, int(m[q])) for q in range(w.n_ranks)]
    pl = oracle.plan(w.n_ranks, w.n_local_experts, w.top_k, r.topk_ids, 2)
    Y, Yd = oracle.expert_rows(oracle.BF16, vals[2]["A"], vals[2]["W"], pl.expert_offsets, w.K,
                               w.N, exact=True)
    A = torch.from_numpy(vals[2]["A"].view(np.int16)).view(torch.bfloat16).double().numpy()
    W = torch.from_numpy(vals[2]["W"].view(np.int16)).view(torch.bfloat16).double().numpy()
    for e in range(w.n_local_experts):
        lo, hi = pl.expert_offsets[e], pl.expert_offsets[e + 1]
        ref = A[lo:hi] @ W[e].T
        bound = 1e-12 * (np.abs(A[lo:hi]) @ np.abs(W[e]).T)
        assert np.all(np.abs(Yd[lo:hi] - ref) <= bound)
    res = full_pipeline(w, r, vals, epoch=1)
    for d in range(w.n_ranks):
        ref = np.einsum("tj,tjn->tn", r.gates[d].astype(np.float64), res["rows_exact"][d])
        np.testing.assert_allclose(res["out_exact"][d], ref, rtol=1e-12, atol=1e-15)
        # the rounded path stays within 2^-7 of the terms' scale of the exact value
        scale = np.einsum("tj,tjn->tn", r.gates[d].astype(np.float64),
                          np.abs(res["rows_exact"][d]))
        got = oracle.bf16_to_f64(res["out"][d])
        assert np.all(np.abs(got - res["out_exact"][d]) <= 2.0**-7 * scale + 1e-30)


def test_expert_rows_exact_on_small_integers():
    rng = np.random.default_rng(11)
    El, K, N, M = 3, 16, 24, 10
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    W = rng.integers(-3, 4, size=(El, N, K)).astype(np.float32)
    offs = np.array([0, 4, 4, M], np.int32)  # expert 1 is empty
    Y = oracle.expert_rows(oracle.BF16, _torch_bf16_bits(A), _torch_bf16_bits(W), offs, K, N)
    ref = np.concatenate([A[0:4] @ W[0].T, A[4:M] @ W[2].T]).astype(np.float64)
    assert np.abs(ref).max() <= 256  # every partial sum is exact in bf16 range of integers
    np.testing.assert_array_equal(oracle.bf16_to_f64(Y), ref)


def test_expert_rows_fp8_matches_dequantised_matmul():
    w = Workload("fp8_small", 2, 2, 2, 16, 256, 256, "fp8_1d2d", "uniform", "sigmoid_sel", 90)
    r = make_routing(w)
    m = int(rows_per_rank(w, r.topk_ids)[0])
    v = make_rank_values(w, 0, m)
    pl = oracle.plan(w.n_ranks, w.n_local_experts, w.top_k, r.topk_ids, 0)
    Y = oracle.expert_rows(oracle.FP8_1D2D, v["A"], v["W"], pl.expert_offsets, w.K, w.N,
                           a_scales=v["a_scales"], w_scales=v["w_scales"])
    a8 = torch.from_numpy(v["A"]).view(torch.float8_e4m3fn).double().numpy()
    w8 = torch.from_numpy(v["W"]).view(torch.float8_e4m3fn).double().numpy()
    A = a8 * np.repeat(v["a_scales"].astype(np.float64), 128, axis=1)
    sw = np.repeat(np.repeat(v["w_scales"].astype(np.float64), 128, axis=1), 128, axis=2)
    Wd = w8 * sw
    for e in range(w.n_local_experts):
        lo, hi = pl.expert_offsets[e], pl.expert_offsets[e + 1]
        assert _ulp_ok(Y[lo:hi], A[lo:hi] @ Wd[e].T)
        # dropping the weight scales (a plausible slip) is far off
        assert not _ulp_ok(Y[lo:hi], A[lo:hi] @ w8[e].T)


# ----------------------------------------------------- scatter / signalling


def _tiny_full(w=None):
    w = w or WORKLOADS["tiny"]
    r = make_routing(w)
    m = rows_per_rank(w, r.topk_ids)
    vals = [make_rank_values(w, q, int(m[q])) for q in range(w.n_ranks)]
    return w, r, vals, full_pipeline(w, r, vals, epoch=5)


def test_scatter_writes_every_slot_exactly_once():
    w, r, vals, res = _tiny_full()
    assert res["bad"] == 0
    np.testing.assert_array_equal(res["hits"], 1)
    for d in range(w.n_ranks):
        assert not np.any(res["recv"][d].view(np.uint16) == 0xFFFF)


def test_scatter_catches_a_planted_index_slip():
    """Swap (src_idx, src_topk) in the plan: the exactly-once check must fail."""
    w = WORKLOADS["tiny"]
    r = make_routing(w)
    R, k, T = w.n_ranks, w.top_k, w.tokens
    recv = [np.full(T * k * w.msg_bytes, 0xFF, np.uint8) for _ in range(R)]
    hits = np.zeros((R, T * k), np.int32)
    bad = 0
    for q in range(R):
        pl = oracle.plan(R, w.n_local_experts, k, r.topk_ids, q)
        pl.src_info = pl.src_info[:, ::-1].copy()
        Y = np.zeros((pl.m_total, w.N), np.uint16)
        hits, b = oracle.scatter(Y, np.arange(pl.m_total), pl, R, k, w.N, w.msg_bytes, T, recv,
                                 hits)
        bad += b
    assert bad > 0 or np.any(hits != 1)


def test_signal_counts_and_flag_order():
    w, r, vals, res = _tiny_full()
    R, El = w.n_ranks, w.n_local_experts
    ids = r.topk_ids
    for q in range(R):
        log = res["logs"][q]
        np.testing.assert_array_equal(res["counters"][q], El)
        for d in range(R):
            ev = [tuple(x) for x in log if x[2] == d]
            counts = [x for x in ev if x[0] == 0]
            flags = [i for i, x in enumerate(ev) if x[0] == 1]
            assert len(counts) == El and len(flags) == 1
            assert flags[0] == len(ev) - 1  # the flag follows every expert of (q -> d)
            assert ev[flags[0]][3] == El - 1
            for e in range(El):
                routed = int(np.sum(ids[d] == q * El + e))  # brute-force count
                assert res["counts"][d][e * R + q] == routed
            assert res["counts"][d][El * R + q] == 5


def test_per_expert_signal_words_decode_to_the_plan_counts():
    """Default mode: the high half of every count word is the call's epoch, the low
    half the row count the brute-force-pinned plan gives; the flag words stay
    untouched, and a later call re-tags every word."""
    w = WORKLOADS["tiny"]
    r = make_routing(w)
    R, El = w.n_ranks, w.n_local_experts
    bufs = [np.full(El * R + R, np.uint64(0xFFFFFFFFFFFFFFFF), np.uint64) for _ in range(R)]
    for epoch in (7, 2**32 + 3):
        for q in range(R):
            pl = oracle.plan(R, El, w.top_k, r.topk_ids, q)
            log = oracle.signal_per_expert(R, El, q, pl.send_counts, epoch, bufs)
            assert len(log) == El * R and (log[:, 0] == 0).all()
        for d in range(R):
            words = bufs[d][:El * R].reshape(El, R)
            assert ((words >> np.uint64(32)) == np.uint64(epoch & 0xFFFFFFFF)).all()
            for q in range(R):
                keys = _brute_plan(r.topk_ids, R, El, q)
                for e in range(El):
                    n = sum(1 for key in keys if key[0] == e and key[1] == d)
                    assert int(words[e, q] & np.uint64(0xFFFFFFFF)) == n
            assert (bufs[d][El * R:] == np.uint64(0xFFFFFFFFFFFFFFFF)).all()


def test_signal_flag_never_before_last_expert():
    """With a counter already at El-2 for every destination, the first expert
    signalled must not publish the flag; the second must."""
    R, El = 2, 3
    sc = np.ones((El, R), np.int32)
    counts = [np.zeros(El * R + R, np.uint64) for _ in range(R)]
    ctr = np.full(R, El - 2, np.int32)
    log = oracle.signal(R, El, 0, sc, 9, counts, ctr)
    kinds = [(int(x[0]), int(x[1])) for x in log]
    assert (1, 0) not in kinds and (1, 1) in kinds


# ----------------------------------------------------------------- combine


def test_combine_matches_numpy():
    w, r, vals, res = _tiny_full()
    k, N, T = w.top_k, w.N, w.tokens
    for d in range(w.n_ranks):
        rows = oracle.bf16_to_f64(res["recv"][d].view(np.uint16)).reshape(T, k, N)
        ref = np.einsum("tj,tjn->tn", r.gates[d].astype(np.float64), rows)
        assert _ulp_ok(res["out"][d], ref)
        # a transposed gate (slot order reversed) is detected
        bad = np.einsum("tj,tjn->tn", r.gates[d][:, ::-1].astype(np.float64), rows)
        assert not _ulp_ok(res["out"][d], bad)


def test_dense_by_token_crosscheck():
    """out[t] = sum_j g[t,j] * bf16(h[t,j] . W_{e(t,j)}^T), with h looked up by a
    Python loop and the matmul done by numpy; no plan, no scatter."""
    w, r, vals, res = _tiny_full()
    R, El, k, T, N = w.n_ranks, w.n_local_experts, w.top_k, w.tokens, w.N
    keys = {q: _brute_plan(r.topk_ids, R, El, q) for q in range(R)}
    row_of = {q: {(key[1], key[2], key[3]): i for i, key in enumerate(keys[q])} for q in range(R)}
    f64 = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()
    for d in range(R):
        ref = np.zeros((T, N))
        for t in range(T):
            for j in range(k):
                g = int(r.topk_ids[d, t, j])
                q, e = g // El, g % El
                h = f64(vals[q]["A"][row_of[q][(d, t, j)]])
                y = f64(_torch_bf16_bits((h @ f64(vals[q]["W"][e]).T).astype(np.float32)))
                ref[t] += float(r.gates[d, t, j]) * y
        got = oracle.bf16_to_f64(res["out"][d])
        rms = np.sqrt(np.mean(ref**2))
        # two bf16 roundings (row, output) on each side: 2^-7 of max(|ref|, rms)
        assert np.all(np.abs(got - ref) <= 2.0**-7 * np.maximum(np.abs(ref), rms))


def test_identity_weights_move_data_exactly():
    """K = N, W_e = 2^c_e * I, top_k = 1, gate 1: every output row equals its
    token's activation row times 2^c_e, bit for bit."""
    w = Workload("ident", 4, 2, 1, 24, 128, 128, "bf16", "uniform", "softmax_indep", 91)
    r = make_routing(w)
    r.gates[:] = 1.0
    m = rows_per_rank(w, r.topk_ids)
    vals = []
    for q in range(w.n_ranks):
        v = make_rank_values(w, q, int(m[q]))
        eye = np.stack([np.eye(w.N, dtype=np.float32) * 2.0**(e + 1 - q)
                        for e in range(w.n_local_experts)])
        v["W"] = _torch_bf16_bits(eye)
        vals.append(v)
    res = full_pipeline(w, r, vals, epoch=1)
    keys = {q: _brute_plan(r.topk_ids, w.n_ranks, w.n_local_experts, q) for q in range(w.n_ranks)}
    for d in range(w.n_ranks):
        for t in range(w.tokens):
            g = int(r.topk_ids[d, t, 0])
            q, e = g // w.n_local_experts, g % w.n_local_experts
            row = keys[q].index((e, d, t, 0))
            a = oracle.bf16_to_f64(vals[q]["A"][row])
            np.testing.assert_array_equal(oracle.bf16_to_f64(res["out"][d][t]),
                                          a * 2.0**(e + 1 - q))


def test_fp8_identity_weights_move_data_exactly():
    """Blockwise fp8, K = N, W_e = I (e4m3 1.0), power-of-two scales, top_k = 1,
    gate 1: out[t, n] = sa[row, n/128] * sw[e, n/128, n/128] * a8[row, n] exactly
    (a dropped or transposed scale index changes the result)."""
    w = Workload("ident8", 2, 2, 1, 20, 256, 256, "fp8_1d2d", "uniform", "softmax_indep", 92)
    r = make_routing(w)
    r.gates[:] = 1.0
    m = rows_per_rank(w, r.topk_ids)
    rng = np.random.default_rng(3)
    vals = []
    for q in range(w.n_ranks):
        v = make_rank_values(w, q, int(m[q]))
        v["W"] = np.zeros_like(v["W"])
        for e in range(w.n_local_experts):
            np.fill_diagonal(v["W"][e], 0x38)
        v["a_scales"] = np.exp2(rng.integers(-4, 5, v["a_scales"].shape)).astype(np.float32)
        v["w_scales"] = np.exp2(rng.integers(-4, 5, v["w_scales"].shape)).astype(np.float32)
        vals.append(v)
    res = full_pipeline(w, r, vals, epoch=1)
    keys = {q: _brute_plan(r.topk_ids, w.n_ranks, w.n_local_experts, q) for q in range(w.n_ranks)}
    n_blk = np.arange(w.N) // 128
    for d in range(w.n_ranks):
        for t in range(w.tokens):
            g = int(r.topk_ids[d, t, 0])
            q, e = g // w.n_local_experts, g % w.n_local_experts
            row = keys[q].index((e, d, t, 0))
            a8 = torch.from_numpy(vals[q]["A"][row]).view(torch.float8_e4m3fn).double().numpy()
            want = a8 * vals[q]["a_scales"][row, n_blk] * vals[q]["w_scales"][e, n_blk, n_blk]
            np.testing.assert_array_equal(oracle.bf16_to_f64(res["out"][d][t]), want)


def test_dispatch_places_every_token_row_by_the_brute_force_keys():
    w = WORKLOADS["tiny"]
    r = make_routing(w)
    rng = np.random.default_rng(5)
    tokens = [rng.integers(0, 2**16, (w.tokens, 24), dtype=np.uint16) for _ in range(w.n_ranks)]
    for q in range(w.n_ranks):
        pl = oracle.plan(w.n_ranks, w.n_local_experts, w.top_k, r.topk_ids, q)
        A_in = oracle.dispatch(pl, tokens, w.top_k)
        keys = _brute_plan(r.topk_ids, w.n_ranks, w.n_local_experts, q)
        assert A_in.shape[0] == len(keys)
        for m, (_, rk, t, _) in enumerate(keys):
            np.testing.assert_array_equal(A_in[m], tokens[rk][t])


def test_swiglu_matches_an_independent_form_and_special_values():
    """SiLU(x) = x * sigmoid(x) = (x / 2) * (1 + tanh(x / 2)): a second form of the
    same function, evaluated independently; plus values fixed by the definition."""
    rng = np.random.default_rng(8)
    inter = 64
    g32 = (rng.standard_normal((50, inter)) * 4).astype(np.float32)
    u32 = rng.standard_normal((50, inter)).astype(np.float32)
    G = _torch_bf16_bits(np.concatenate([g32, u32], axis=1))
    A = oracle.swiglu(G, inter)
    g = oracle.bf16_to_f64(G[:, :inter])
    u = oracle.bf16_to_f64(G[:, inter:])
    want = oracle.bf16_from_f64(0.5 * g * (1.0 + np.tanh(0.5 * g)) * u)
    diff = np.abs(oracle.bf16_to_f64(A) - oracle.bf16_to_f64(want))
    assert (diff <= 2.0**-8 * np.abs(oracle.bf16_to_f64(want)) + 1e-30).all()
    assert (A == want).mean() > 0.999  # the two forms round alike except at rare ties
    # the gate selects: SiLU(0) = 0; SiLU(large) ~ large; SiLU(-large) ~ 0; the up half scales
    G2 = _torch_bf16_bits(np.array([[0.0, 30.0, -30.0, 1.0, 3.0, 3.0, 3.0, 0.0]], np.float32))
    A2 = oracle.bf16_to_f64(oracle.swiglu(G2, 4))[0]
    assert A2[0] == 0.0 and A2[3] == 0.0
    assert abs(A2[1] - 90.0) <= 0.5 and abs(A2[2]) < 1e-9


def _bf16_rne_f64(x: np.ndarray) -> np.ndarray:
    """Round float64 values (normal bf16 range) to the nearest bf16 value, ties to
    even, as float64: 8 significant bits, written out from the definition."""
    m, e = np.frexp(np.asarray(x, np.float64))  # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def test_swiglu_exact_matches_an_independent_form_and_special_values():
    """The activation of the unrounded products (the epilogue form): SiLU(g) * u with
    SiLU(x) = (x / 2) * (1 + tanh(x / 2)), evaluated independently in float64 and
    rounded once to bf16 by a separate restatement of round-to-nearest-even."""
    rng = np.random.default_rng(18)
    inter = 96
    g = rng.standard_normal((40, inter)) * 4
    u = rng.standard_normal((40, inter))
    G = np.concatenate([g, u], axis=1)  # float64, not bf16-representable
    A = oracle.bf16_to_f64(oracle.swiglu_exact(G, inter))
    want = _bf16_rne_f64(0.5 * g * (1.0 + np.tanh(0.5 * g)) * u)
    assert (np.abs(A - want) <= 2.0**-8 * np.abs(want) + 1e-30).all()
    assert (A == want).mean() > 0.999  # the two forms round alike except at rare ties
    # rounding G to bf16 first (the separate-pass form) is a different result
    A_rounded_first = oracle.bf16_to_f64(oracle.swiglu(oracle.bf16_from_f64(G), inter))
    assert (A_rounded_first != A).mean() > 0.05
    exact = g / (1.0 + np.exp(-g)) * u
    assert np.abs(A - exact).mean() < np.abs(A_rounded_first - exact).mean()
    # the up half scales the result exactly (power of two); SiLU(0) = 0; the gate
    # half is the one that goes through SiLU (swapping the halves changes the result)
    A2 = oracle.bf16_to_f64(oracle.swiglu_exact(np.concatenate([g, 2 * u], axis=1), inter))
    np.testing.assert_array_equal(A2, 2 * A)
    G3 = np.array([[0.0, -30.0, 5.0, 1.5, 5.0, -30.0]])
    A3 = oracle.bf16_to_f64(oracle.swiglu_exact(G3, 3))[0]
    assert A3[0] == 0.0
    assert abs(A3[1]) < 1e-9  # SiLU(-30) * 5 ~ -4.7e-12
    assert A3[2] == _bf16_rne_f64(np.array([5.0 / (1.0 + np.exp(-5.0)) * -30.0]))[0]


def test_sampled_pipeline_agrees_with_full():
    w, r, vals, res = _tiny_full()
    toks = np.array([0, 5, 63, 17])
    s = sampled_pipeline(w, r, lambda q: vals[q], 2, toks)
    np.testing.assert_array_equal(s["out"], res["out"][2][toks])
    rows = res["recv"][2].view(np.uint16).reshape(w.tokens, w.top_k, w.N)
    np.testing.assert_array_equal(s["rows"], rows[toks])
