"""Failure paths on the GPU, made without faulting it: a flag that nothing
sets (the bounded wait must run out and report EP_STATUS_TIMEOUT, and the
context must stay usable), and a destination outside the receive buffer
(EP_STATUS_BOUNDS, that row skipped, every other row delivered)."""

import numpy as np
import pytest
import torch

import moe_expert_gemm_gb300 as ep
from parity_util import build_system, make_inputs
from synth import WORKLOADS

pytestmark = pytest.mark.gpu


def test_combine_times_out_when_a_producer_never_ran():
    w = WORKLOADS["tiny"]
    routing, values = make_inputs(w)
    s = build_system(w, routing, values)
    s.timeout_ns = 50_000_000  # 50 ms
    for r in range(w.n_ranks):
        if r != 3:
            s.send(r, epoch=1)
    s.out[0].zero_()
    s.combine(0, epoch=1)
    torch.cuda.synchronize()
    st = s.status_words()
    assert st[2] & ep.EP_STATUS_TIMEOUT
    assert int(s.out[0].view(torch.int16).abs().sum()) == 0  # nothing combined
    # the context is still usable: the missing producer runs, the combine succeeds
    s.status.zero_()
    s.send(3, epoch=1)
    s.combine(0, epoch=1)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    assert int(s.out[0].view(torch.int16).abs().sum()) > 0


def test_out_of_range_destination_is_skipped_and_reported():
    w = WORKLOADS["tiny"]
    routing, values = make_inputs(w)
    s = build_system(w, routing, values)
    r = 1
    si = s.plans[r]["src_info"]
    bad_row = 5
    t_bad, j_bad = (int(x) for x in si[bad_row].tolist())
    si[bad_row, 0] = w.tokens  # src_idx past max_tokens_per_rank
    s.send(r, epoch=1)
    torch.cuda.synchronize()
    st = s.status_words()
    assert st[1] & ep.EP_STATUS_BOUNDS
    # every other row of rank 1 arrived; the bad row's slot still holds the sentinel
    pl = s.plan_host(r)
    seg = pl["seg_offsets"]
    e = int(np.searchsorted(pl["expert_offsets"], bad_row, side="right") - 1)
    dst = int(np.searchsorted(seg[e], bad_row, side="right") - 1)
    for m in range(pl["m_total"]):
        e_m = int(np.searchsorted(pl["expert_offsets"], m, side="right") - 1)
        d_m = int(np.searchsorted(seg[e_m], m, side="right") - 1)
        t, j = pl["src_info"][m]
        if m == bad_row:
            t, j = t_bad, j_bad
        row = s.recv[d_m].view(torch.int16)[(t * w.top_k + j) * w.N:(t * w.top_k + j + 1) * w.N]
        written = bool((row != -1).any())
        assert written == (m != bad_row), m
    assert dst >= 0


@pytest.mark.parametrize("kind", ["end_past_rows", "non_monotone"])
def test_malformed_expert_offsets_are_clamped(kind):
    """A corrupted plan's expert row ranges are made monotone and clamped to the rows
    of A: expert e runs over [o_e, o_{e+1}) with o_e = min(max(0, raw_0 .. raw_e),
    max_rows). Rows that then lie outside every destination segment of their expert
    are skipped with EP_STATUS_BOUNDS; every other row arrives as in an intact call,
    every count word and the rank flag are published, and nothing waits out."""
    w = WORKLOADS["tiny"]
    routing, values = make_inputs(w)
    r = 1
    good = build_system(w, routing, values)
    good.send(r, epoch=1)
    s = build_system(w, routing, values)
    s.set_operands(r, values[r]["A"], values[r]["W"], pad_rows=64)  # rows past m_total
    eo = s.plans[r]["expert_offsets"]
    raw = eo.cpu().numpy().copy()
    max_rows = int(s.send_args(r, 1).max_rows)
    assert max_rows > raw[-1] + 5
    if kind == "end_past_rows":
        raw[-1] = max_rows + 1000  # rows [m_total, max_rows) join the last expert
        skipped_experts = set()
    else:
        raw[1] = raw[2] + 5  # expert 0 would end past expert 1, which becomes empty
        skipped_experts = {1}
    eo.copy_(torch.from_numpy(raw))
    s.send(r, epoch=1)
    torch.cuda.synchronize()
    st = s.status_words()
    assert st[1] & ep.EP_STATUS_BOUNDS
    assert not st[1] & ep.EP_STATUS_TIMEOUT
    for d in range(w.n_ranks):
        np.testing.assert_array_equal(s.counts[d].cpu().numpy(), good.counts[d].cpu().numpy())
    pl = good.plan_host(r)
    seg = pl["seg_offsets"]
    for m in range(pl["m_total"]):
        e = int(np.searchsorted(pl["expert_offsets"], m, side="right") - 1)
        d = int(np.searchsorted(seg[e], m, side="right") - 1)
        t, j = (int(x) for x in pl["src_info"][m])
        sl = slice((t * w.top_k + j) * w.N, (t * w.top_k + j + 1) * w.N)
        got = s.recv[d].view(torch.int16)[sl].cpu()
        if e in skipped_experts:
            assert bool((got == -1).all()), m
        else:
            assert torch.equal(got, good.recv[d].view(torch.int16)[sl].cpu()), m
