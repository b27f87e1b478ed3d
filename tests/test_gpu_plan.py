"""The plan kernel on its own (GPU): bit-exact against the oracle's plan over
routings that cut each source rank's entries into several chunks, ragged chunk
ends, every rank count; malformed routing and capacity overflow reported through
the status word, never a fault."""

import numpy as np
import pytest
import torch

import moe_expert_gemm_gb300 as ep
import oracle
from moe_expert_gemm_gb300.system import EpSystem
from parity_util import assert_plan_equal
from synth import Workload, make_routing

pytestmark = pytest.mark.gpu


def _system(R, El, k, T):
    return EpSystem(R, El, k, T, 128, 128, "bf16")


@pytest.mark.parametrize("R,El,k,T,law", [
    (1, 3, 1, 77, "uniform"),        # one rank: 32 chunks of 3 entries
    (3, 5, 2, 1001, "zipf"),         # 10 chunks per rank, 2 spare warps, ragged ends
    (5, 7, 3, 333, "biased"),
    (8, 32, 8, 8192, "uniform"),     # the decode / fp8 routing shape
    (8, 16, 8, 2048, "zipf"),        # skewed, empty experts
    (8, 256, 1, 64, "uniform"),      # many local experts, most of them empty
])
def test_plan_matches_oracle(R, El, k, T, law):
    w = Workload("plan", R, El, k, T, 128, 128, "bf16", law, "softmax_sel", 70)
    routing = make_routing(w)
    s = _system(R, El, k, T)
    s.set_routing(routing.topk_ids)
    for r in range(R):
        s.plan(r)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    for r in range(R):
        assert_plan_equal(s.plan_host(r), oracle.plan(R, El, k, routing.topk_ids, r))


def test_out_of_range_expert_ids_are_reported_and_skipped():
    R, El, k, T = 4, 2, 2, 50
    w = Workload("plan_bad", R, El, k, T, 128, 128, "bf16", "uniform", "softmax_sel", 71)
    ids = make_routing(w).topk_ids.copy()
    ids[1, 7, 0] = R * El      # past the last expert
    ids[2, 9, 1] = -1
    s = _system(R, El, k, T)
    s.set_routing(ids)
    for r in range(R):
        s.status.zero_()
        s.plan(r)
        torch.cuda.synchronize()
        assert s.status_words()[0] & ep.EP_STATUS_ROUTING
        # a malformed entry is routed nowhere: the plan equals that of a routing
        # where it points at an expert of another rank
        fixed = ids.copy()
        other = ((r + 1) % R) * El
        fixed[1, 7, 0] = other
        fixed[2, 9, 1] = other
        assert_plan_equal(s.plan_host(r), oracle.plan(R, El, k, fixed, r))


def test_capacity_overflow_publishes_an_empty_plan():
    R, El, k, T = 4, 2, 2, 64
    w = Workload("plan_cap", R, El, k, T, 128, 128, "bf16", "uniform", "softmax_sel", 72)
    routing = make_routing(w)
    s = _system(R, El, k, T)
    s.set_routing(routing.topk_ids)
    need = oracle.plan(R, El, k, routing.topk_ids, 0).m_total
    p = s.plan(0, max_rows=need - 1)
    torch.cuda.synchronize()
    assert s.status_words()[0] & ep.EP_STATUS_CAPACITY
    assert int(p["m_total"].item()) == 0
    assert int(p["expert_offsets"].abs().sum()) == 0
    assert int(p["send_counts"].abs().sum()) == 0
    s.status.zero_()
    p = s.plan(0, max_rows=need)  # exactly enough
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    assert int(p["m_total"].item()) == need
