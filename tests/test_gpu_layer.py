"""A whole MoE layer on the library's kernels (GPU): dispatch of the routed token
rows, the up/gate projection (the grouped GEMM with the sink disabled, K = H,
N = 2I), the gated activation, the fused down-projection + send and the combine.

Every kernel is compared with the oracle on the inputs that kernel actually got:
the gathered rows bit-exact against the oracle's dispatch; the up/gate rows within
1e-2 of the oracle's (bf16 output, fp32 accumulation in another order); the
activation within one bf16 ulp (2^-7 relative) of the oracle's activation of the
GPU's own G (fp32 SiLU rounded once, against float64 rounded once), or, with the
activation in the up/gate GEMM's epilogue, within 1e-2 of the oracle's activation
of the exact products (the fp32 accumulation order is the only other source); the
down-projection, the send, the signalling and the combine as in the other parity
tests, against the oracle's pipeline fed the GPU's A."""

import numpy as np
import pytest
import torch

from moe_expert_gemm_gb300.system import EpSystem
import oracle
from oracle.pipeline import full_pipeline, layer_pipeline
from parity_util import TOL, assert_combine_close, max_rel_err
from synth import Workload, WORKLOADS, make_layer_values, make_routing

pytestmark = pytest.mark.gpu

LAYER_CASES = [
    ("tiny", WORKLOADS["tiny"]),
    # several row blocks per expert (CTA pairs for the 512-wide up/gate GEMM), empty
    # experts under zipf routing, eight ranks
    ("zipf_pairs", Workload("layer_zipf", 4, 3, 2, 400, 256, 384, "bf16", "zipf",
                            "softmax_sel", 80)),
    ("eight_ranks", Workload("layer_r8", 8, 2, 2, 64, 128, 256, "bf16", "biased",
                             "softmax_sel", 81)),
]


@pytest.mark.parametrize("fused_act", [False, True], ids=["separate_act", "fused_act"])
@pytest.mark.parametrize("name,w", LAYER_CASES, ids=[c[0] for c in LAYER_CASES])
def test_layer_parity(name, w, fused_act):
    routing = make_routing(w)
    lv = [make_layer_values(w, r) for r in range(w.n_ranks)]
    s = EpSystem(w.n_ranks, w.n_local_experts, w.top_k, w.tokens, w.K, w.N, "bf16")
    s.set_routing(routing.topk_ids)
    for r in range(w.n_ranks):
        s.plan(r)
        s.set_layer_operands(r, lv[r]["X"], lv[r]["W1"], lv[r]["W2"])
        s.set_gates(r, routing.gates[r])
    for r in range(w.n_ranks):
        s.layer_forward(r, epoch=3, fused_act=fused_act)
    for d in range(w.n_ranks):
        s.combine(d, epoch=3)
    torch.cuda.synchronize()
    assert (s.status_words() == 0).all(), s.status_words()
    ref = layer_pipeline(w, routing, lv, epoch=3)
    gpu_A = []
    for r in range(w.n_ranks):
        m = ref["plans"][r].m_total
        bits = lambda t: t[:m].view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(bits(s.layer[r]["A_in"]), ref["A_in"][r])
        A = bits(s.ops[r]["A"])
        if fused_act:
            # no G: the epilogue applies the activation to the fp32 accumulators; the
            # oracle applies it to the exact products (one bf16 rounding each)
            pl = ref["plans"][r]
            _, Gd = oracle.expert_rows(oracle.BF16, ref["A_in"][r], lv[r]["W1"],
                                       pl.expert_offsets, w.N, 2 * w.K, exact=True)
            assert max_rel_err(A, oracle.swiglu_exact(Gd, w.K)) <= TOL["bf16"], r
        else:
            G = bits(s.layer[r]["G"])
            assert max_rel_err(G, ref["G"][r]) <= TOL["bf16"], r
            assert max_rel_err(A, oracle.swiglu(G, w.K)) <= 2.0**-7, r
        gpu_A.append({"A": A, "W": lv[r]["W2"]})
    down = full_pipeline(w, routing, gpu_A, epoch=3)
    for d in range(w.n_ranks):
        np.testing.assert_array_equal(s.counts[d].cpu().numpy().view(np.uint64),
                                      down["counts"][d])
        got = s.recv[d].cpu().numpy().view(np.uint16)
        assert max_rel_err(got, down["recv"][d].view(np.uint16)) <= TOL["bf16"], d
        out = s.out[d].view(torch.int16).cpu().numpy().view(np.uint16)
        assert_combine_close(out, down["out"][d], down["out_exact"][d], down["rows_exact"][d],
                             routing.gates[d], TOL["bf16"], (w.name, "layer", d))
