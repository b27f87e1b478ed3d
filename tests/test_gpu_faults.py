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
