"""The producer and consumer calls captured once in a CUDA graph and replayed:
every launch reads its operands through the pointers it was captured with, so
new operand values written in place between replays give the oracle's results
for those values (counts, flags, received rows and combined outputs). The calls
allocate nothing and never synchronise, which is what capture requires."""

import dataclasses

import numpy as np
import pytest
import torch

from oracle.pipeline import full_pipeline
from parity_util import TOL, assert_combine_close, build_system, make_inputs, max_rel_err
from synth import WORKLOADS, Workload

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny", WORKLOADS["tiny"]),  # single-CTA kernel
    ("pairs", Workload("graph_pairs", 2, 2, 2, 600, 256, 512, "bf16", "uniform",
                       "softmax_sel", 75)),  # CTA pairs: T*top_k/E_l >= 256
    ("fp8", Workload("graph_fp8", 4, 2, 2, 64, 256, 256, "fp8_1d2d", "uniform",
                     "sigmoid_sel", 76)),
]


def _upload_in_place(s, r, v):
    ops = s.ops[r]
    m = v["A"].shape[0]
    if s.dtype == "bf16":
        ops["A"][:m].view(torch.int16).copy_(torch.from_numpy(np.ascontiguousarray(v["A"]).view(np.int16)))
        ops["W"].view(torch.int16).copy_(torch.from_numpy(np.ascontiguousarray(v["W"]).view(np.int16)))
    else:
        ops["A"][:m].copy_(torch.from_numpy(np.ascontiguousarray(v["A"])))
        ops["W"].copy_(torch.from_numpy(np.ascontiguousarray(v["W"])))
        ops["a_scales"][:m].copy_(torch.from_numpy(np.ascontiguousarray(v["a_scales"], dtype=np.float32)))
        ops["w_scales"].copy_(torch.from_numpy(np.ascontiguousarray(v["w_scales"], dtype=np.float32)))


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_send_and_combine_replayed_from_a_cuda_graph(name, w):
    routing, values = make_inputs(w)
    s = build_system(w, routing, values)
    epoch = 5
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):  # one eager pass on the capture stream first
        for r in range(w.n_ranks):
            s.send(r, epoch, stream=stream)
        for d in range(w.n_ranks):
            s.combine(d, epoch, stream=stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        cs = torch.cuda.current_stream()
        for r in range(w.n_ranks):
            s.send(r, epoch, stream=cs)
        for d in range(w.n_ranks):
            s.combine(d, epoch, stream=cs)
    torch.cuda.synchronize()

    for rep in range(2):
        # new operand values (another seed, same routing) written through the captured pointers
        w2 = dataclasses.replace(w, wid=w.wid + 100 + rep)
        values2 = make_inputs(w2, routing)[1]
        for r in range(w.n_ranks):
            _upload_in_place(s, r, values2[r])
        for d in range(w.n_ranks):
            s.recv[d].fill_(0xFF)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert (s.status_words() == 0).all()
        ref = full_pipeline(w, routing, values2, epoch=epoch)
        tol = TOL[w.dtype]
        for d in range(w.n_ranks):
            np.testing.assert_array_equal(s.counts[d].cpu().numpy().view(np.uint64), ref["counts"][d])
            assert max_rel_err(s.recv[d].cpu().numpy().view(np.uint16),
                               ref["recv"][d].view(np.uint16)) <= tol, (rep, d)
            out = s.out[d].view(torch.int16).cpu().numpy().view(np.uint16)
            assert_combine_close(out, ref["out"][d], ref["out_exact"][d], ref["rows_exact"][d],
                                 routing.gates[d], tol, (w.name, "graph", rep, d))
