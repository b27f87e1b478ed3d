"""The N > 1 host path of bench.py on CPU: two processes over gloo (no GPU).

N GPUs run N independent replicas: each process plays logical rank
(rank mod n_ranks), the step time is the maximum over processes, the value is
the whole job's tokens over that time, and the reference arm runs (and prints)
on rank 0 only."""

import io
import os
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got_rank, _, got_world = bench.dist_env()
        step_ms = [2.0, 3.5][rank]  # rank 1 is the slower replica
        slowest = bench.max_over_ranks(step_ms, world, "cpu")
        dist.barrier()
        # the reference arm under torchrun: only rank 0 does work and prints
        out = io.StringIO()
        if rank != 0:
            with redirect_stdout(out):
                bench.run_reference(argparse_ns(), rank, world)
        q.put(dict(rank=rank, env=(got_rank, got_world), replica=bench.replica_rank(rank, 8),
                   slowest=slowest,
                   value=bench.job_tokens_per_s(world, 4096, slowest),
                   ref_out=out.getvalue()))
    finally:
        dist.destroy_process_group()


def argparse_ns():
    import argparse
    return argparse.Namespace(workload="tiny", steps=1, warmup=0)


def test_two_replicas_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in procs), key=lambda d: d["rank"])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r["env"] for r in res] == [(0, 2), (1, 2)]
    assert [r["replica"] for r in res] == [0, 1]
    assert all(r["slowest"] == 3.5 for r in res)  # every rank sees the maximum
    assert all(abs(r["value"] - 2 * 4096 / 3.5e-3) < 1e-6 for r in res)
    assert res[1]["ref_out"] == ""  # rank 1 of the reference arm prints nothing


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.replica_rank(9, 8) == 1
    assert bench.replica_rank(3, 8, first=6) == 1  # replicas start from the timed rank
    assert bench.job_tokens_per_s(1, 1000, 2.0) == 500_000.0


def test_reference_arm_line_on_rank_0():
    """The reference arm's JSON line (the oracle on the host, tiny workload): the keys
    a harness reads, its cpu_baseline describing the run, and an e2e equal to it."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    out = io.StringIO()
    with redirect_stdout(out):
        args = bench.parse_args(["--impl", "reference", "--workload", "tiny", "--steps", "2",
                                 "--warmup", "1", "--rank", "1"])
        bench.run_reference(args, 0, 1)
    line = json.loads(out.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s"
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["config"]["workload"] == "tiny" and line["config"]["my_rank"] == 1
    # the same config the GPU arm prints for these arguments, key for key
    from synth import WORKLOADS, make_routing, rows_per_rank
    w = WORKLOADS["tiny"]
    rows = rows_per_rank(w, make_routing(w).topk_ids)
    assert line["config"] == bench.config_dict(w, 1, int(rows[1]), args, 1)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert "rank 1" in cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def _ipc_worker(rank, world, port, q):
    """Handle exchange of the one-rank-per-process path over gloo, with stand-in
    handles and a stand-in import (no GPU): each rank's table holds its own
    addresses at its own index and what it imported from every peer elsewhere."""
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from moe_expert_gemm_gb300 import ep_ipc_handle
    from moe_expert_gemm_gb300.peers import handle_bytes, handle_from_bytes, peer_tables
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = []
        for kind in range(2):  # receive buffer, receive-count buffer
            h = ep_ipc_handle()
            h.handle[0], h.handle[63] = rank, kind
            h.offset, h.bytes = 4096 * (rank + 1) + kind, 1 << 20
            mine.append(handle_bytes(h))
        gathered = [None] * world
        dist.all_gather_object(gathered, tuple(mine))
        imported = []

        def fake_import(b):
            h = handle_from_bytes(b)
            imported.append((h.handle[0], h.handle[63], h.offset))
            return 10_000 * (h.handle[0] + 1) + 100 * h.handle[63] + h.offset % 4096
        own = (111 + rank, 222 + rank)
        tables = peer_tables(rank, own, gathered, fake_import)
        q.put(dict(rank=rank, tables=tables, imported=sorted(imported)))
    finally:
        dist.destroy_process_group()


def test_ipc_handle_exchange_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29800 + os.getpid() % 1000
    procs = [ctx.Process(target=_ipc_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in procs), key=lambda d: d["rank"])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # rank 0: its own buffers at index 0, rank 1's imported (kind k -> 20000 + 100k + k)
    assert res[0]["tables"] == [[111, 20_000 + 0 + 0], [222, 20_000 + 100 + 1]]
    assert res[1]["tables"] == [[10_000 + 0 + 0, 112], [10_000 + 100 + 1, 223]]
    # each rank imported exactly its peer's two handles, with their offsets
    assert res[0]["imported"] == [(1, 0, 8192), (1, 1, 8193)]
    assert res[1]["imported"] == [(0, 0, 4096), (0, 1, 4097)]


def test_peer_tables_reject_mismatched_exports():
    import pytest
    sys.path.insert(0, ROOT)
    from moe_expert_gemm_gb300.peers import handle_from_bytes, peer_tables
    with pytest.raises(ValueError):
        peer_tables(2, (1, 2), [(b"a", b"b"), (b"c", b"d")], lambda b: 0)
    with pytest.raises(ValueError):
        peer_tables(0, (1, 2), [(b"a", b"b"), (b"c",)], lambda b: 0)
    with pytest.raises(ValueError):
        handle_from_bytes(b"short")
