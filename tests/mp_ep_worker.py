"""One rank of an expert-parallel group run as separate processes on one GPU (the
worker of test_gpu_multiprocess.py; not a test module).

Each process owns its rank's receive buffers, maps its peers' through CUDA IPC
handles exchanged over gloo, runs its own fused send and its own combine, and saves
what it received and combined for the parent to compare with the oracle.

Every rank goes through the same fixed sequence of phases, each closed by a
barrier, whatever happened before: a rank that hit an error skips its GPU calls
but keeps its buffers allocated and keeps taking part in the barriers, so no
process frees memory a peer's send may still store into. Every producer kernel
has completed (synchronised, then a barrier) before any combine is launched, so no
kernel of one process waits on a kernel of another that is still running; the one
wait that runs out (the "stopped rank" phase) waits for a flag nothing will set.
"""

from __future__ import annotations

import datetime
import os
import sys
import traceback

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)

STOP_EPOCH = 3
STOP_TIMEOUT_NS = 50_000_000  # 50 ms


def run_rank(rank: int, world: int, port: int, wspec: tuple, signal_mode: int, outdir: str):
    for p in (ROOT, TESTS):
        if p not in sys.path:
            sys.path.insert(0, p)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np
    import torch
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=300))
    errors: list = []
    ep = None

    def phase(fn):
        if errors:
            return
        try:
            fn()
        except Exception:  # recorded; the rank keeps taking part in the barriers
            errors.append(traceback.format_exc())

    def save(tag):
        def _save():
            torch.cuda.synchronize()
            np.savez(os.path.join(outdir, f"rank{rank}_{tag}.npz"),
                     recv=ep.recv.cpu().numpy(), counts=ep.counts.cpu().numpy().view(np.uint64),
                     out=ep.out.view(torch.int16).cpu().numpy().view(np.uint16),
                     status=ep.status_words(),
                     peers_mapped=np.array([int(x != 0) for x in ep.recv_ptrs]))
        phase(_save)

    try:
        from moe_expert_gemm_gb300.peers import EpRank
        from synth import Workload, make_rank_values, make_routing, rows_per_rank

        w = Workload(*wspec)
        routing = make_routing(w)
        rows = rows_per_rank(w, routing.topk_ids)

        def setup():
            nonlocal ep
            torch.cuda.set_device(0)
            v = make_rank_values(w, rank, int(rows[rank]))
            ep = EpRank(w.n_ranks, rank, w.n_local_experts, w.top_k, w.tokens, w.K, w.N, w.dtype,
                        signal_mode=signal_mode)
            ep.set_routing(routing.topk_ids)
            ep.plan()
            ep.set_operands(v["A"], v["W"], v.get("a_scales"), v.get("w_scales"))
            ep.set_gates(routing.gates[rank])
            torch.cuda.synchronize()
        phase(setup)
        # the handle exchange is a collective: every rank takes part
        gathered = [None] * world
        mine = None
        if not errors:
            try:
                mine = ep.export_handles()
            except Exception:
                errors.append(traceback.format_exc())
        dist.all_gather_object(gathered, mine)
        if any(g is None for g in gathered):
            errors.append("a rank exported no handles")
        phase(lambda: ep.attach(gathered))
        dist.barrier()

        for epoch in (1, 2, STOP_EPOCH):
            stop = epoch == STOP_EPOCH
            phase(lambda: (ep.reset_buffers(), ep.out.zero_(), torch.cuda.synchronize()))
            dist.barrier()  # every buffer reset before any producer stores into it
            if not (stop and rank == world - 1):  # the last rank stops sending
                phase(lambda: (ep.send(epoch), torch.cuda.synchronize()))
            dist.barrier()  # every producer kernel has completed
            phase(lambda: (ep.combine(epoch, timeout_ns=STOP_TIMEOUT_NS if stop else None),
                           torch.cuda.synchronize()))
            save(f"epoch{epoch}")
            dist.barrier()
    finally:
        # no process unmaps or frees before every process is done with the GPU
        try:
            dist.barrier()
        except Exception:
            errors.append(traceback.format_exc())
        if ep is not None:
            try:
                ep.close()
            except Exception:
                errors.append(traceback.format_exc())
        try:
            dist.barrier()
        except Exception:
            errors.append(traceback.format_exc())
        with open(os.path.join(outdir, f"rank{rank}.err"), "w") as f:
            f.write("\n".join(errors))
        dist.destroy_process_group()
