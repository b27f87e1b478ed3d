"""grouped_gemm_combine_send_noalloc, the entry point for callers that cannot
allocate device memory (hosts that own every allocation and forbid cudaMalloc in
their per-call path): through the C ABI, calls in a row must give what the
allocating entry point gives -- the same received rows (within the parity
tolerance) and the same count and flag words, bit for bit -- also when calls of
different shapes (other expert and rank counts, the CTA-pair kernel) take turns
on the one shared counter array, and without the device memory in use growing.

This file is collected last on purpose, so that a failure here cannot hide the
results of the other GPU tests in a run that stops at the first failure.
"""

import numpy as np
import pytest
import torch

import moe_expert_gemm_gb300 as ep
from parity_util import TOL, build_system, make_inputs, max_rel_err
from synth import WORKLOADS, Workload

pytestmark = pytest.mark.gpu

# more local experts and ranks than the tiny workload, 256-row pair tiles
PAIR_SHAPE = Workload("noalloc_pairs", 8, 16, 8, 512, 256, 512, "bf16", "zipf", "softmax_sel", 91)


def _reference(w, r):
    """The system of workload w, and what the allocating entry point delivers for
    producer rank r (receive buffers, count words)."""
    routing, values = make_inputs(w)
    s = build_system(w, routing, values)
    s.send(r, epoch=1)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    recv = [b.cpu().numpy().copy() for b in s.recv]
    counts = [c.cpu().numpy().view(np.uint64).copy() for c in s.counts]
    return s, recv, counts


def _noalloc_call(s, r, epoch):
    s.reset_buffers()
    args = s.send_args(r, epoch)
    args.atomic_counter = None  # ignored by this entry point
    args.rank_completion_counter = None
    ep.grouped_gemm_combine_send_noalloc(s.cfg(r), args)


def _check(s, w, r, epoch, ref_recv, ref_counts):
    assert (s.status_words() == 0).all(), s.status_words()
    flag = w.n_local_experts * w.n_ranks + r
    for d in range(w.n_ranks):
        got = s.recv[d].cpu().numpy().view(np.uint16)
        ref = ref_recv[d].view(np.uint16)
        sent = ref != 0xFFFF  # slots this producer writes; the rest keep the sentinel
        np.testing.assert_array_equal(got != 0xFFFF, sent)
        assert max_rel_err(got[sent], ref[sent]) <= TOL["bf16"]
        want = ref_counts[d].copy()
        want[flag] = epoch
        np.testing.assert_array_equal(s.counts[d].cpu().numpy().view(np.uint64), want)


def test_noalloc_matches_allocating_entry_point_twice():
    w = WORKLOADS["tiny"]
    r = 2
    s, ref_recv, ref_counts = _reference(w, r)
    for epoch in (1, 2):
        _noalloc_call(s, r, epoch)
        torch.cuda.synchronize()
        _check(s, w, r, epoch, ref_recv, ref_counts)


def test_noalloc_shapes_take_turns_on_the_shared_array_without_allocating():
    w1, r1 = WORKLOADS["tiny"], 1
    w2, r2 = PAIR_SHAPE, 5
    s1, recv1, counts1 = _reference(w1, r1)
    s2, recv2, counts2 = _reference(w2, r2)
    # first calls on this device (the module holding the array may load now)
    _noalloc_call(s1, r1, 1)
    _noalloc_call(s2, r2, 1)
    torch.cuda.synchronize()
    used = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for epoch in (2, 3):
        _noalloc_call(s1, r1, epoch)
        torch.cuda.synchronize()
        _check(s1, w1, r1, epoch, recv1, counts1)
        _noalloc_call(s2, r2, epoch)
        torch.cuda.synchronize()
        _check(s2, w2, r2, epoch, recv2, counts2)
    # the calls themselves allocate nothing: torch's allocator holds what it held,
    # and the device has as much free memory as before
    assert torch.cuda.memory_allocated() == used
    assert torch.cuda.mem_get_info()[0] == free_before


def test_noalloc_rejects_sizes_beyond_its_array():
    cfg = ep.ep_config(2, 0, ep.EP_MAX_LOCAL_EXPERTS + 1, 2, 8, 8, 128, 128, 256, ep.EP_BF16, -1)
    code = ep.raw_call("grouped_gemm_combine_send_noalloc", cfg, ep.ep_send_args(), None)
    assert code == ep.EP_ERR_UNSUPPORTED
