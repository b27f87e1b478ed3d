"""Expert parallelism with one rank per process (GPU): every logical rank is its own
process on one GPU, with its own receive buffers; the ranks
exchange CUDA IPC handles of those buffers over gloo, map their peers' buffers, and
each runs its own fused send into the mapped peer memory and its own combine
("ep_signal_completion": direct memory access to a device on the same node;
"P3PeerSendConfig": one receive-buffer pointer per rank).

Compared with the oracle, bit for bit for count and flag words and within the
tolerance for rows and combined outputs, on two epochs in a row; then the last rank
stops sending (its process stays, so its buffers stay mapped) and every combine's
bounded wait runs out with EP_STATUS_TIMEOUT, leaving the outputs that need the
stopped rank unwritten (with per-expert signals, the other tokens are combined).
"""

import dataclasses
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import mp_ep_worker as worker
from oracle.pipeline import SENTINEL_WORD, full_pipeline
from parity_util import TOL, assert_combine_close, make_inputs, max_rel_err
from synth import WORKLOADS, Workload

pytestmark = pytest.mark.gpu

EP_STATUS_TIMEOUT = 0x2
STATUS_SEND, STATUS_COMBINE = 1, 2

CASES = [
    ("tiny_rank_flag", WORKLOADS["tiny"], 0),
    ("tiny_per_expert", WORKLOADS["tiny"], 1),
    # eight processes, 256-row CTA-pair tiles, Zipf routing
    ("pairs_8_ranks", Workload("mp_pairs", 8, 16, 8, 512, 256, 512, "bf16", "zipf",
                               "softmax_sel", 92), 0),
    # blockwise fp8 operands (the fp8 kernel's bulk-copy rows into mapped peer memory)
    ("fp8_rank_flag", Workload("mp_fp8", 4, 2, 2, 100, 256, 256, "fp8_1d2d", "uniform",
                               "sigmoid_sel", 93), 0),
]


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_group(w, signal_mode, outdir):
    ctx = mp.get_context("spawn")
    port = _free_port()
    spec = dataclasses.astuple(w)
    procs = [ctx.Process(target=worker.run_rank,
                         args=(r, w.n_ranks, port, spec, signal_mode, str(outdir)))
             for r in range(w.n_ranks)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
    stuck = [p for p in procs if p.is_alive()]
    for p in stuck:
        p.kill()
        p.join()
    assert not stuck, "a rank process did not finish"
    errs = []
    for r in range(w.n_ranks):
        with open(os.path.join(outdir, f"rank{r}.err")) as f:
            e = f.read().strip()
        if e:
            errs.append(f"rank {r}:\n{e}")
    assert not errs, "\n".join(errs)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]


def _load(outdir, rank, epoch):
    return dict(np.load(os.path.join(outdir, f"rank{rank}_epoch{epoch}.npz")))


@pytest.mark.parametrize("name,w,signal_mode", CASES, ids=[c[0] for c in CASES])
def test_ranks_as_processes_match_the_oracle(name, w, signal_mode, tmp_path):
    _run_group(w, signal_mode, tmp_path)
    routing, values = make_inputs(w)
    tol = TOL[w.dtype]
    R, El = w.n_ranks, w.n_local_experts
    for epoch in (1, 2):
        ref = full_pipeline(w, routing, values, epoch=epoch, per_expert=bool(signal_mode))
        for d in range(R):
            got = _load(tmp_path, d, epoch)
            assert (got["peers_mapped"] == 1).all()
            assert (got["status"] == 0).all(), (epoch, d, got["status"])
            np.testing.assert_array_equal(got["counts"], ref["counts"][d])
            assert max_rel_err(got["recv"].view(np.uint16), ref["recv"][d].view(np.uint16)) <= tol
            assert_combine_close(got["out"], ref["out"][d], ref["out_exact"][d],
                                 ref["rows_exact"][d], routing.gates[d], tol,
                                 (name, "processes", epoch, d))

    # the last rank stopped sending: its words stay unwritten, every other producer's
    # are there, and the combines gave up
    stopped = R - 1
    epoch = worker.STOP_EPOCH
    ref = full_pipeline(w, routing, values, epoch=epoch, per_expert=bool(signal_mode))
    needs_stopped = routing.topk_ids // El == stopped  # [R][T][k]
    for d in range(R):
        got = _load(tmp_path, d, epoch)
        assert got["status"][STATUS_COMBINE] & EP_STATUS_TIMEOUT, (d, got["status"])
        assert got["status"][STATUS_SEND] == 0
        words = got["counts"]
        for r in range(R):
            mine = [e * R + r for e in range(El)] + ([El * R + r] if signal_mode == 0 else [])
            if r == stopped:
                assert (words[mine] == SENTINEL_WORD).all(), (d, r)
            else:
                np.testing.assert_array_equal(words[mine], ref["counts"][d][mine])
        waits = needs_stopped[d].any(axis=1) if signal_mode else np.ones(w.tokens, bool)
        assert (got["out"][waits] == 0).all()
        if (~waits).any():
            assert_combine_close(got["out"][~waits], ref["out"][d][~waits],
                                 ref["out_exact"][d][~waits], ref["rows_exact"][d][~waits],
                                 routing.gates[d][~waits], tol, (name, "stopped rank", d))
