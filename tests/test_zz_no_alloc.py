"""grouped_gemm_combine_send_noalloc, the entry point for callers that cannot
allocate device memory (hosts that own every allocation and forbid cudaMalloc in
their per-call path): through the C ABI, two calls in a row must give what the
allocating entry point gives -- the same received rows (within the parity
tolerance) and the same count and flag words, bit for bit.

This file is collected last on purpose, so that a failure here cannot hide the
results of the other GPU tests in a run that stops at the first failure.
"""

import numpy as np
import pytest
import torch

import moe_expert_gemm_gb300 as ep
from parity_util import TOL, build_system, make_inputs, max_rel_err
from synth import WORKLOADS

pytestmark = pytest.mark.gpu


def test_noalloc_matches_allocating_entry_point_twice():
    w = WORKLOADS["tiny"]
    routing, values = make_inputs(w)
    s = build_system(w, routing, values)
    r = 2
    s.send(r, epoch=1)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all()
    ref_recv = [b.cpu().numpy().copy() for b in s.recv]
    ref_counts = [c.cpu().numpy().view(np.uint64).copy() for c in s.counts]
    flag = w.n_local_experts * w.n_ranks + r

    for epoch in (1, 2):
        s.reset_buffers()
        args = s.send_args(r, epoch)
        args.atomic_counter = None  # ignored by this entry point
        args.rank_completion_counter = None
        ep.grouped_gemm_combine_send_noalloc(s.cfg(r), args)
        torch.cuda.synchronize()
        assert (s.status_words() == 0).all(), s.status_words()
        for d in range(w.n_ranks):
            got = s.recv[d].cpu().numpy().view(np.uint16)
            ref = ref_recv[d].view(np.uint16)
            sent = ref != 0xFFFF  # slots this producer writes; the rest keep the sentinel
            np.testing.assert_array_equal(got != 0xFFFF, sent)
            assert max_rel_err(got[sent], ref[sent]) <= TOL["bf16"]
            want = ref_counts[d].copy()
            want[flag] = epoch
            np.testing.assert_array_equal(s.counts[d].cpu().numpy().view(np.uint64), want)


def test_noalloc_rejects_sizes_beyond_its_array():
    cfg = ep.ep_config(2, 0, ep.EP_MAX_LOCAL_EXPERTS + 1, 2, 8, 8, 128, 128, 256, ep.EP_BF16, -1)
    code = ep.raw_call("grouped_gemm_combine_send_noalloc", cfg, ep.ep_send_args(), None)
    assert code == ep.EP_ERR_UNSUPPORTED
