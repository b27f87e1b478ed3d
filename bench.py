#!/usr/bin/env python
"""Benchmark: fused expert-GEMM + combine-scatter step of one logical EP rank.

One step = the whole hot path of one rank on its own batch: the grouped
down-projection GEMM whose epilogue sends every row to its token's rank
(grouped_gemm_combine_send, with the completion signalling), then the
gate-weighted combine of the rank's own tokens (ep_combine_reduce). The other
logical ranks' receive buffers are separate allocations in the same HBM; their
producers run once, untimed, before the timed region, and before every step a
single fill writes their rank flags for the new epoch (the stand-in for peers
finishing on their own GPUs).

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]

Under torchrun each process plays one logical rank (RANK mod n_ranks) on its own
GPU, independently: replicas with no collective on the data path ("weak"
scaling); the barrier and max-over-ranks timing use torch.distributed.

The default workload is the Mixtral-like prefill (8 ranks x 1 expert, top-2,
4096 tokens per rank, 14336 -> 4096 bf16). Every step's inputs (A of that rank:
~235 MB, its expert weight: ~117 MB) exceed the 129 MB L2, so no explicit flush
is needed between steps; workloads whose per-step inputs fit in L2 flush it
outside the timed events with a 512 MB write followed by a read of the same
buffer (cold L2 without dirty lines left for the timed kernel to write back).

``--impl reference`` times the CPU oracle (the plain C restatement of the path)
on bounded token samples of the same workload, on the host's cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused expert-GEMM+combine-scatter tokens/s; TFLOP/s and % of roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 10**6


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral_prefill")
    ap.add_argument("--rank", default="0",
                    help="logical rank timed at N=1 (replicas start from it): an index, or "
                         "'max' for the rank that receives the most rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target host time of the CPU-baseline sample")
    ap.add_argument("--trace", default=None,
                    help="after timing, run one traced send and write its summary here")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override tokens per rank (profiling a smaller case of a workload)")
    ap.add_argument("--path", choices=["fused", "unfused", "layer"], default="fused",
                    help="unfused: the comparator without the sink (GEMM rows to a local C, "
                         "then ep_scatter_send); layer: a whole MoE layer (dispatch, up/gate "
                         "GEMM, activation, the fused down-projection + send, combine; bf16)")
    ap.add_argument("--layer-act", choices=["fused", "separate"], default="fused",
                    help="--path layer: the activation in the up/gate GEMM's epilogue (fused) "
                         "or as its own pass over the GEMM's rows (separate)")
    ap.add_argument("--overlap", action="store_true",
                    help="launch the combine (and, for --path layer, the two GEMMs) as a "
                         "programmatic dependent that starts while the kernel before it "
                         "finishes; the per-kernel times then come from a serialised copy of "
                         "every timed step, run right after it")
    ap.add_argument("--signal-mode", choices=["rank_flag", "per_expert"], default="rank_flag",
                    help="completion signalling: ep_ord_r rank flags (default) or per-expert "
                         "count words with a per-token wait in the combine")
    ap.add_argument("--send-warps", type=int, default=-1, choices=[-1, 0, 4],
                    help="sink placement: -1 library choice, 0 inside the output warps, "
                         "4 dedicated send warps (bf16)")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the per-workload measurements (every workload's rank 0 and "
                         "most-loaded rank) that follow the headline at N=1")
    ap.add_argument("--pw-steps", type=int, default=30,
                    help="timed steps of each per-workload measurement")
    ap.add_argument("--solo", action="store_true",
                    help="profiling aid: only the timed rank's operands, no peer staging, and "
                         "the step is the fused send alone (no combine, no e2e, no baseline)")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class NvmlClocks:
    """Read-only NVML queries (ctypes on NVIDIA's libnvidia-ml) of one GPU's SM
    clock, clock-event reasons and power: sampled every ~2 ms on a thread while a
    timed region runs. Nothing is ever set."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        import ctypes
        import threading
        self.ct, self.threading = ctypes, threading
        self.lib = self.handle = None
        self.samples = []
        self.thread = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            self.lib = lib
            self.handle = self._find_handle(device_index)
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self.reasons_fn = reasons or lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            self.lib = None
        if self.handle is None:
            self.lib = None

    def _find_handle(self, device_index: int):
        import torch
        ct = self.ct
        props = torch.cuda.get_device_properties(device_index)
        h = ct.c_void_p()
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            u = str(uuid)
            u = u if u.startswith("GPU-") else "GPU-" + u
            if self.lib.nvmlDeviceGetHandleByUUID(u.encode(), ct.byref(h)) == 0:
                return h
        if hasattr(props, "pci_bus_id"):
            bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                        props.pci_device_id)
            if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ct.byref(h)) == 0:
                return h
        return None

    @property
    def ok(self) -> bool:
        return self.lib is not None

    def read(self):
        ct = self.ct
        mhz, reasons, mw = ct.c_uint(0), ct.c_ulonglong(0), ct.c_uint(0)
        self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(mhz))  # NVML_CLOCK_SM
        self.reasons_fn(self.handle, ct.byref(reasons))
        self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw))
        return time.perf_counter(), mhz.value, reasons.value, mw.value / 1e3

    def max_sm_mhz(self):
        v = self.ct.c_uint(0)
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, self.ct.byref(v))
        return v.value

    def start(self):
        if not self.ok:
            return
        self.samples = []
        self.stop_flag = False

        def loop():
            while not self.stop_flag:
                self.samples.append(self.read())
                time.sleep(0.002)
        self.thread = self.threading.Thread(target=loop, daemon=True)
        self.thread.start()

    def stop(self, busy=None):
        """Summary of the samples; ``busy`` (t0, t1) perf_counter bounds keep only the
        samples taken while the GPU was known to be running the timed work."""
        if not self.ok or self.thread is None:
            return None
        self.stop_flag = True
        self.thread.join()
        rows = self.samples
        if busy is not None:
            rows = [r for r in rows if busy[0] <= r[0] <= busy[1]] or rows
        if not rows:
            return None
        reasons = sorted({name for r in rows for bit, name in self.REASONS.items()
                          if r[2] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in rows),
                "sm_mhz_min": min(r[1] for r in rows), "sm_max_mhz": self.max_sm_mhz(),
                "power_w_max": max(r[3] for r in rows), "reasons": reasons,
                "samples": len(rows), "source": "NVML, read-only, every ~2 ms in-process"}


class ClockSampler:
    """nvidia-smi sampling (100 ms) of SM clocks and throttle reasons: the fallback
    when NVML cannot be loaded in-process."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, busy=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows), "source": "nvidia-smi every 100 ms"}


def clock_sampler(device_index: int):
    s = NvmlClocks(device_index)
    return s if s.ok else ClockSampler(device_index)


# Sources that decide what the fused GEMM+send kernels do on the device: the kernels,
# their shared headers, and the host code that picks the kernel, tile and tile order.
FUSED_KERNEL_SOURCES = ("ep_api.cu", "ep_gemm_send.cu", "ep_gemm_send_fp8.cu",
                        "ep_gemm_send_pair.cu", "ep_internal.h", "ep_ptx.cuh", "ep_sink.cuh")


def _code_only(text: str) -> str:
    """C++ source without its comments and blank lines (a comment edit does not
    change what a measurement describes)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_sha() -> str:
    """Digest of the fused kernels' code (a measurement taken on other code does not
    describe the current kernels)."""
    csrc = os.path.join(ROOT, "moe_expert_gemm_gb300", "csrc")
    h = hashlib.sha256()
    for name in FUSED_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` from a committed ncu summary, if it was
    taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(workload, {}).get(kernel)
    if not rec or rec.get("source_sha") != kernel_source_sha():
        return None
    return rec.get("bytes_per_launch")


def algorithmic_work(w, plan_counts: np.ndarray, m_rows: int):
    """FLOPs and bytes per launch of the two kernels (per logical rank)."""
    elem = 1 if w.dtype == "fp8_1d2d" else 2
    nonempty = int((plan_counts.sum(axis=1) > 0).sum())
    flops = 2.0 * m_rows * w.K * w.N
    send_bytes = m_rows * w.K * elem + nonempty * w.N * w.K * elem + m_rows * w.N * 2
    if w.dtype == "fp8_1d2d":
        send_bytes += m_rows * (w.K // 128) * 4 + nonempty * (w.N // 128) * (w.K // 128) * 4
    comb_bytes = w.tokens * w.top_k * w.N * 2 + w.tokens * w.N * 2 + w.tokens * w.top_k * 4
    return flops, float(send_bytes), float(comb_bytes)


FLUSH_TEXT = ("flushed before every step: a 512 MB write, then a read of the same buffer "
              "(the timed kernel starts with a cold L2 that holds no dirty lines)")


def flush_l2(buf, e: int):
    """Evict the step's inputs from L2: write a buffer larger than L2, then read it
    back, so that the written-back dirty lines are the flush's cost and not the timed
    kernel's."""
    buf.fill_(e & 0xFF)
    buf.max()


def l2_policy(w, rows_q: int) -> tuple[bool, str]:
    """Whether every step flushes L2, and the config text saying so: the step's
    operand bytes (A of the timed rank and its experts' W) against twice the L2."""
    elem = 1 if w.dtype == "fp8_1d2d" else 2
    step_bytes = rows_q * w.K * elem + w.n_local_experts * w.N * w.K * elem
    if step_bytes < 2 * L2_BYTES:
        return True, FLUSH_TEXT
    return False, f"per-step inputs {step_bytes / 1e6:.0f} MB > L2"


def config_dict(w, q: int, rows_q: int, args, world: int) -> dict:
    """The workload description both arms print (same keys, same values)."""
    return {"workload": w.name, "n_ranks": w.n_ranks, "n_local_experts": w.n_local_experts,
            "top_k": w.top_k, "tokens_per_rank": w.tokens, "K": w.K, "N": w.N,
            "operands": w.dtype, "my_rank": q, "rows": int(rows_q),
            "send_warps": args.send_warps, "path": args.path,
            "combine_overlaps_send": bool(args.overlap and args.path != "unfused"),
            "signal_mode": args.signal_mode, "l2": l2_policy(w, rows_q)[1],
            "parallelism": "replicas: one logical rank per GPU" if world > 1
            else "one logical rank"}


def roofline(w, flops: float, nbytes: float, dom_s: float, peaks: dict, peak_src: str,
             traffic=None) -> dict:
    """Roofline entry of one kernel: tensor-bound when its FLOPs at the tensor peak
    take longer than its bytes at the HBM peak, else HBM-bound."""
    peak_tf = float(peaks["bf16_tflops"]) * (2.0 if w.dtype == "fp8_1d2d" else 1.0)
    peak_bw = float(peaks["hbm_gbs"])
    if flops / (peak_tf * 1e12) >= nbytes / (peak_bw * 1e9):
        tf = flops / dom_s / 1e12
        roof = {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": tf / peak_tf, "traffic": traffic}
    else:
        gbs = nbytes / dom_s / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": peak_bw, "unit": "GB/s",
                "frac": gbs / peak_bw, "traffic": traffic}
    roof["peak_source"] = (f"{peak_src}: " + ("bf16_tflops (burst)" if roof["bound"] == "tensor"
                                              else "hbm_gbs")
                           + (" x2 nominal fp8/bf16 ratio" if w.dtype == "fp8_1d2d"
                              and roof["bound"] == "tensor" else ""))
    return roof


def measure_workload(name: str, steps: int, warmup: int, peaks: dict, peak_src: str,
                     device_index: int, probe_s: float = 0.5) -> dict:
    """Fused send and combine of rank 0 and of the most-loaded rank of one workload,
    every rank staged as in the headline step (serialised kernels, CUDA events on the
    launching stream, L2 flushed between steps where the inputs fit in it, clocks
    sampled), then, after both, a back-to-back probe of each under clock sampling."""
    import torch
    from moe_expert_gemm_gb300.system import EpSystem
    from synth import WORKLOADS, make_rank_values, make_routing, rows_per_rank

    w = WORKLOADS[name]
    routing = make_routing(w)
    rows = rows_per_rank(w, routing.topk_ids)
    qmax = int(np.argmax(rows))
    targets = [0] if qmax == 0 else [0, qmax]
    s = EpSystem(w.n_ranks, w.n_local_experts, w.top_k, w.tokens, w.K, w.N, w.dtype)
    s.set_routing(routing.topk_ids)
    for r in range(w.n_ranks):
        s.plan(r)
        v = make_rank_values(w, r, int(rows[r]))
        s.set_operands(r, v["A"], v["W"], v.get("a_scales"), v.get("w_scales"))
        del v
    for q in targets:
        s.set_gates(q, routing.gates[q])
    for r in range(w.n_ranks):
        s.send(r, epoch=1)
    torch.cuda.synchronize()
    if s.status_words().any():
        raise SystemExit(f"{name}: device status after staging: {s.status_words()}")
    stream = torch.cuda.current_stream()
    epoch = [2]

    def stepper(q):
        """The step of rank q (flush where the inputs fit in L2, the peers' flags, the
        send, the combine), with events around the send and the combine."""
        peer_idx = torch.tensor([w.n_local_experts * w.n_ranks + r for r in range(w.n_ranks)
                                 if r != q], dtype=torch.int64, device="cuda")
        need_flush = l2_policy(w, int(rows[q]))[0]
        flush = torch.empty(512 * 2**20, dtype=torch.uint8, device="cuda") if need_flush else None

        def step(ev=None):
            e = epoch[0]
            epoch[0] += 1
            if flush is not None:
                flush_l2(flush, e)
            if peer_idx.numel():
                s.counts[q].index_fill_(0, peer_idx, e)
            if ev is not None:
                ev[0].record(stream)
            s.send(q, e, stream)
            if ev is not None:
                ev[1].record(stream)
            s.combine(q, e, stream)
            if ev is not None:
                ev[2].record(stream)
        return step

    out = {}
    # every target's timed steps first (each after a short idle gap, so that no earlier
    # sustained run holds the clocks down), then the sustained probes
    for q in targets:
        plan_q = s.plan_host(q)
        m_rows = plan_q["m_total"]
        flops, send_bytes, comb_bytes = algorithmic_work(w, plan_q["send_counts"], m_rows)
        step = stepper(q)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        time.sleep(0.2)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        clk = clock_sampler(device_index)
        clk.start()
        t0 = time.perf_counter()
        for i in range(steps):
            step(evs[i])
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        timed_clocks = clk.stop(busy=(t0, t1))
        send_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
        comb_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
        roof = roofline(w, flops, send_bytes, send_ms / 1e3, peaks, peak_src,
                        measured_traffic(w.name, "grouped_gemm_combine_send") if q == 0 else None)
        out["rank0" if q == 0 else "max_rank"] = {
            "rank": q, "rows": int(m_rows), "steps": steps, "warmup": warmup,
            "fused_ms": send_ms, "combine_ms": comb_ms, "step_ms": send_ms + comb_ms,
            "tokens_per_s": w.tokens / ((send_ms + comb_ms) / 1e3),
            "tflops": flops / (send_ms / 1e3) / 1e12,
            "combine_gbs": comb_bytes / (comb_ms / 1e3) / 1e9,
            "roofline": roof, "l2": l2_policy(w, m_rows)[1], "clocks": timed_clocks}
        if timed_clocks and timed_clocks.get("sm_mhz"):
            # the kernel's time in SM clock cycles (thousands) at the median clock sampled
            timed_clocks["fused_kcycles_at_median_clock"] = send_ms * timed_clocks["sm_mhz"]
    for q in targets:
        # the same step back to back for ~probe_s, under clock sampling
        step = stepper(q)
        clk = clock_sampler(device_index)
        clk.start()
        probe = []
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < probe_s and len(probe) < 20000:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            step(ev)
            probe.append(ev)
            if len(probe) % 64 == 0:
                probe[-64][2].synchronize()  # keep the queue short
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        clocks = clk.stop(busy=(t0, t1))
        probe_send = statistics.mean(e[0].elapsed_time(e[1]) for e in probe)
        entry = out["rank0" if q == 0 else "max_rank"]
        entry["probe"] = {"seconds": t1 - t0, "steps": len(probe), "fused_ms": probe_send,
                          "clocks": clocks}
        if clocks and clocks.get("sm_mhz"):
            entry["probe"]["fused_kcycles_at_median_clock"] = probe_send * clocks["sm_mhz"]
    if s.status_words().any():
        raise SystemExit(f"{name}: device status after timing: {s.status_words()}")
    del s
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------- oracle arm

def cpu_sample(w, routing, values, dst: int, target_s: float, plans: dict):
    """Time the oracle on a token sample of destination `dst`; returns
    (tokens/s, threads, description)."""
    import oracle
    from oracle.pipeline import sampled_pipeline

    rng = np.random.default_rng(123)
    order = rng.permutation(w.tokens)
    # calibrate on a growing probe: tiny samples under-use the threads
    n = min(w.tokens, 16)
    while True:
        t0 = time.perf_counter()
        sampled_pipeline(w, routing, lambda r: values[r], dst, order[:n], plans=plans)
        dt = time.perf_counter() - t0
        if dt >= 0.2 * target_s or n >= w.tokens:
            break
        n = min(w.tokens, n * 4)
    per_tok = max(dt / n, 1e-9)
    n = int(min(w.tokens, max(4, target_s / per_tok)))
    toks = np.sort(order[:n])
    t0 = time.perf_counter()
    sampled_pipeline(w, routing, lambda r: values[r], dst, toks, plans=plans)
    dt = time.perf_counter() - t0
    desc = (f"{n} of rank {dst}'s {w.tokens} tokens: their {w.top_k} expert rows each "
            f"(GEMM rows from every producer rank) and their combine, {dt:.1f} s")
    return n / dt, oracle.default_threads(), desc, n, dt


# ----------------------------------------------------------- multi-process host logic
# N > 1 runs N independent replicas (one logical rank per GPU, no data-path
# collective): each process plays logical rank (rank mod n_ranks), the timed
# region is bracketed by barriers, the step time is the maximum over processes
# and the reported value is the whole job's tokens over that time.

def replica_rank(rank: int, n_ranks: int, first: int = 0) -> int:
    """The logical rank a process plays (process 0 plays `first`)."""
    return (first + rank) % n_ranks


def max_over_ranks(x: float, world: int, device) -> float:
    """The maximum of x over all processes (x itself when there is one)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_replica: int, step_ms: float) -> float:
    """Whole-job throughput: every replica's tokens over the slowest replica's step."""
    return world * tokens_per_replica / (step_ms / 1e3)


def run_reference(args, rank, world):
    if rank != 0:
        return
    from synth import WORKLOADS, make_rank_values, make_routing, rows_per_rank
    import oracle

    w = WORKLOADS[args.workload]
    routing = make_routing(w)
    rows = rows_per_rank(w, routing.topk_ids)
    q = int(np.argmax(rows)) if args.rank == "max" else int(args.rank)
    if not 0 <= q < w.n_ranks:
        raise SystemExit(f"--rank must name a logical rank below {w.n_ranks}")
    values = [make_rank_values(w, r, int(rows[r])) for r in range(w.n_ranks)]
    plans = {r: oracle.plan(w.n_ranks, w.n_local_experts, w.top_k, routing.topk_ids, r)
             for r in range(w.n_ranks)}
    budget = max(0.1, 150.0 / max(1, args.steps + args.warmup))  # whole run ~ 2.5 minutes
    from oracle.pipeline import sampled_pipeline
    rng = np.random.default_rng(7)
    probe = min(w.tokens, 16)
    t0 = time.perf_counter()
    sampled_pipeline(w, routing, lambda r: values[r], q, rng.permutation(w.tokens)[:probe],
                     plans=plans)
    per_tok = max((time.perf_counter() - t0) / probe, 1e-9)
    n = int(min(w.tokens, max(1, budget / per_tok)))
    times = []
    for i in range(args.warmup + args.steps):
        toks = np.sort(rng.permutation(w.tokens)[:n])
        t0 = time.perf_counter()
        sampled_pipeline(w, routing, lambda r: values[r], q, toks, plans=plans)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    step_s = sum(times) / len(times)
    value = n / step_s
    cores = oracle.default_threads()
    sample = (f"each step: {n} of rank {q}'s {w.tokens} tokens, their {w.top_k} rows each "
              f"(GEMM from every producer rank) and their combine")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, q, int(rows[q]), args, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- GPU arm

def main():
    args = parse_args()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    import moe_expert_gemm_gb300 as ep
    from moe_expert_gemm_gb300.system import EpSystem
    from synth import WORKLOADS, make_layer_values, make_rank_values, make_routing, rows_per_rank

    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    ep.load()

    w = WORKLOADS[args.workload]
    if args.tokens:
        import dataclasses
        w = dataclasses.replace(w, tokens=args.tokens, name=f"{w.name}@T{args.tokens}")
    routing = make_routing(w)
    rows = rows_per_rank(w, routing.topk_ids)
    first = int(np.argmax(rows)) if args.rank == "max" else int(args.rank)
    if not 0 <= first < w.n_ranks:
        raise SystemExit(f"--rank must name a logical rank below {w.n_ranks}")
    q = replica_rank(rank, w.n_ranks, first)  # the logical rank this process plays
    ranks = [q] if args.solo else list(range(w.n_ranks))
    layer = args.path == "layer"
    if layer and (w.dtype != "bf16" or args.solo):
        raise SystemExit("--path layer runs bf16 workloads with every rank staged")
    values = {r: (make_layer_values(w, r) if layer else make_rank_values(w, r, int(rows[r])))
              for r in ranks}

    s = EpSystem(w.n_ranks, w.n_local_experts, w.top_k, w.tokens, w.K, w.N, w.dtype,
                 send_warps=args.send_warps,
                 signal_mode=1 if args.signal_mode == "per_expert" else 0)
    s.set_routing(routing.topk_ids)
    for r in ranks:
        s.plan(r)
        v = values[r]
        if layer:
            s.set_layer_operands(r, v["X"], v["W1"], v["W2"])
        else:
            s.set_operands(r, v["A"], v["W"], v.get("a_scales"), v.get("w_scales"))
    s.set_gates(q, routing.gates[q])
    # peers' rows land in every receive buffer once (their producers are not timed)
    for r in ranks:
        if layer:
            s.layer_forward(r, epoch=1, fused_act=args.layer_act == "fused")
        else:
            s.send(r, epoch=1)
    torch.cuda.synchronize()
    st = s.status_words()
    if st.any():
        raise SystemExit(f"device status after staging: {st}")
    plan_q = s.plan_host(q)
    m_rows = plan_q["m_total"]
    flops, send_bytes, comb_bytes = algorithmic_work(w, plan_q["send_counts"], m_rows)

    stream = torch.cuda.current_stream()
    peer_idx = torch.tensor([w.n_local_experts * w.n_ranks + r for r in range(w.n_ranks)
                             if r != q], dtype=torch.int64, device="cuda")
    # per-expert signalling: the peers' count words of rank q's buffer, (rk, e) ->
    # e*R + rk, each holding the rows rank rk's expert e sends to q (from the routing)
    peers = [rk for rk in range(w.n_ranks) if rk != q]
    ids_q = routing.topk_ids[q].reshape(-1)
    pe_idx = torch.tensor([e * w.n_ranks + rk for rk in peers for e in range(w.n_local_experts)],
                          dtype=torch.int64, device="cuda")
    pe_rows = torch.tensor([int((ids_q == rk * w.n_local_experts + e).sum()) for rk in peers
                            for e in range(w.n_local_experts)], dtype=torch.int64, device="cuda")

    def publish_peers(e: int):
        """Stand-in for the other ranks finishing on their own GPUs."""
        if args.signal_mode == "per_expert":
            if pe_idx.numel():
                s.counts[q].index_copy_(0, pe_idx, pe_rows + ((e & 0xFFFFFFFF) << 32))
        elif peer_idx.numel():
            s.counts[q].index_fill_(0, peer_idx, e)
    step_bytes = int(s.ops[q]["A"].numel() * s.ops[q]["A"].element_size()
                     + s.ops[q]["W"].numel() * s.ops[q]["W"].element_size())
    need_flush = step_bytes < 2 * L2_BYTES if layer else l2_policy(w, m_rows)[0]
    flush = torch.empty(512 * 2**20, dtype=torch.uint8, device="cuda") if need_flush else None
    epoch = [2]
    unfused = args.path == "unfused"
    C_local = s.local_C(q) if unfused else None

    # the combine may start while the fused send finishes (its rows are ordered by the
    # flags it acquires, not by the kernel boundary); the per-kernel breakdown is taken
    # from separately timed steps with the two kernels serialised
    overlap = args.overlap and not unfused

    def one_step(evs=None, serial=False):
        e = epoch[0]
        epoch[0] += 1
        if flush is not None:
            flush_l2(flush, e)
        publish_peers(e)
        if evs is not None:
            evs[0].record(stream)
        if layer:
            inner = evs is not None and (serial or not overlap)
            s.layer_forward(q, e, stream, events=[evs[4], evs[5], evs[6], evs[7]] if inner
                            else None, fused_act=args.layer_act == "fused",
                            overlap=overlap and not serial)
        elif unfused:
            s.send(q, e, stream, p3_control=-1, C=C_local)
            if evs is not None:
                evs[3].record(stream)
            ep.ep_scatter_send(s.cfg(q), s.scatter_args(q, e, C_local), stream)
        else:
            s.send(q, e, stream)
        if evs is not None and (serial or not overlap):
            evs[1].record(stream)
        if not args.solo:
            # the kernel before the combine is the send, which writes none of its inputs
            s.combine(q, e, stream, overlap=ep.EP_OVERLAP_INPUTS_READY
                      if overlap and not serial else ep.EP_OVERLAP_NONE)
        if evs is not None:
            evs[2].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = clock_sampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.05 if isinstance(clocks, NvmlClocks) else 0.5)  # sampler running first
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    # with overlap, every timed step is followed by the same step with its kernels
    # serialised, which gives the per-kernel times under the same clocks and power
    serial_events = ([[torch.cuda.Event(enable_timing=True) for _ in range(8)]
                      for _ in range(args.steps)] if overlap else None)
    torch.cuda.synchronize()
    t_busy0 = time.perf_counter()
    for i in range(args.steps):
        one_step(events[i])
        if overlap:
            one_step(serial_events[i], serial=True)
    torch.cuda.synchronize()
    t_busy1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    step_overlapped = (statistics.mean(e[0].elapsed_time(e[2]) for e in events)
                       if overlap else None)
    if overlap:
        events = serial_events
    clk = clocks.stop(busy=(t_busy0, t_busy1))
    send_ms = [e[0].elapsed_time(e[1]) for e in events]
    comb_ms = [e[1].elapsed_time(e[2]) for e in events]
    gemm_ms = [e[0].elapsed_time(e[3]) for e in events] if unfused else None
    if layer:  # dispatch, up/gate GEMM, activation, fused down-projection + send
        stage_ms = [statistics.mean(e[a].elapsed_time(e[b]) for e in events)
                    for a, b in ((0, 4), (4, 5), (5, 6), (6, 7))]
    step_ms = step_overlapped if overlap else sum(a + b for a, b in zip(send_ms, comb_ms)) / args.steps
    st = s.status_words()
    if st.any():
        raise SystemExit(f"device status after timing: {st}")

    if args.trace and rank == 0:
        from moe_expert_gemm_gb300.system import summarize_trace
        e = epoch[0]
        epoch[0] += 1
        publish_peers(e)
        tr = s.send_traced(q, e, records=256)
        if not args.solo:
            s.combine(q, e, stream)
        torch.cuda.synchronize()
        with open(args.trace, "w") as f:
            json.dump({"workload": w.name, "summary": summarize_trace(tr), "blocks": tr}, f)

    # ------------------------------------------------------ end to end (host buffers)
    # Every step copies its inputs (A, the fp8 scales, the gates) from pinned host memory
    # and reads its output back, through the same public calls. The kernels of a step
    # run in order on one stream; the copies run on their own streams with inputs and
    # outputs double-buffered, so step i+1's host->device copies overlap step i's kernels
    # and step i's read-back overlaps step i+1's.
    e2e = None
    if not args.no_e2e and not args.solo and not unfused and not layer:
        ops = s.ops[q]
        A_bufs = [ops["A"], torch.empty_like(ops["A"])]
        fp8 = "a_scales" in ops
        sa_bufs = [ops["a_scales"], torch.empty_like(ops["a_scales"])] if fp8 else [None, None]
        g_bufs = [s.gates[q], torch.empty_like(s.gates[q])]
        o_bufs = [s.out[q], torch.empty_like(s.out[q])]
        A_host = ops["A"].cpu().pin_memory()
        sa_host = ops["a_scales"].cpu().pin_memory() if fp8 else None
        g_host = s.gates[q].cpu().pin_memory()
        out_host = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in o_bufs]
        h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
        inputs_free = [None, None]  # compute of the last step that used each input slot
        out_free = [None, None]     # read-back of the last step that used each output slot
        cfg_q = s.cfg(q)

        def e2e_step(i):
            b = i % 2
            e = epoch[0]
            epoch[0] += 1
            if inputs_free[b] is not None:
                h2d_stream.wait_event(inputs_free[b])
            with torch.cuda.stream(h2d_stream):
                A_bufs[b].copy_(A_host, non_blocking=True)
                if fp8:
                    sa_bufs[b].copy_(sa_host, non_blocking=True)
                g_bufs[b].copy_(g_host, non_blocking=True)
                h2d_done = h2d_stream.record_event()
            stream.wait_event(h2d_done)
            if out_free[b] is not None:
                stream.wait_event(out_free[b])
            publish_peers(e)
            a = s.send_args(q, e)
            a.A = ep.ptr(A_bufs[b])
            if fp8:
                a.a_scales = ep.ptr(sa_bufs[b])
            ep.grouped_gemm_combine_send(cfg_q, a, stream)
            ep.ep_combine_reduce(cfg_q, s.combine_args(
                q, e, gates=g_bufs[b], out=o_bufs[b],
                overlap=ep.EP_OVERLAP_INPUTS_READY if overlap else ep.EP_OVERLAP_NONE), stream)
            inputs_free[b] = stream.record_event()
            d2h_stream.wait_event(inputs_free[b])
            with torch.cuda.stream(d2h_stream):
                out_host[b].copy_(o_bufs[b], non_blocking=True)
                out_free[b] = d2h_stream.record_event()

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)
        d2h_stream.wait_event(e0)
        for i in range(args.steps):
            e2e_step(args.warmup + i)
        stream.wait_stream(d2h_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.steps
        h2d = A_host.numel() * A_host.element_size() + g_host.numel() * 4
        if fp8:
            h2d += sa_host.numel() * 4
        e2e = {"value": w.tokens / (e2e_ms / 1e3), "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(out_host[0].numel() * out_host[0].element_size()),
               "pipeline": "two-deep: a step's host-to-device copies overlap the previous "
                           "step's kernels, its read-back the next step's"}
        # the read-back of the last step equals the device-timed step's output
        last = out_host[(args.warmup + args.steps - 1) % 2]
        if not torch.equal(last.view(torch.int16), s.out[q].cpu().view(torch.int16)):
            raise SystemExit("end-to-end output differs from the device-timed output")
        if world > 1:
            e2e["value"] = job_tokens_per_s(world, w.tokens,
                                            max_over_ranks(e2e_ms, world, "cuda"))
        if s.status_words().any():
            raise SystemExit(f"device status after e2e: {s.status_words()}")

    step_ms = max_over_ranks(step_ms, world, "cuda")

    peaks, peak_src = load_peaks()
    send_s = statistics.mean(send_ms) / 1e3
    comb_s = statistics.mean(comb_ms) / 1e3
    # the dominant kernel: the fused GEMM + send, (unfused) the GEMM into the local C, or
    # (layer) the up/gate GEMM
    if layer:
        flops = 2.0 * m_rows * w.N * 2 * w.K
        send_bytes = m_rows * w.N * 2 + plan_q["send_counts"].shape[0] * 2 * w.K * w.N * 2 \
            + m_rows * (1 if args.layer_act == "fused" else 2) * w.K * 2
        dom_s = stage_ms[1] / 1e3
    else:
        dom_s = statistics.mean(gemm_ms) / 1e3 if unfused else send_s
    tflops = flops / dom_s / 1e12
    traffic = None if unfused or layer else measured_traffic(w.name, "grouped_gemm_combine_send")
    roof = roofline(w, flops, send_bytes, dom_s, peaks, peak_src, traffic)
    roof["kernel"] = ("grouped_gemm_combine_send with the sink disabled (rows to a local C)"
                      if unfused else "the up/gate grouped GEMM (K = H, N = 2I, rows to a "
                      "local buffer)" if layer else "grouped_gemm_combine_send")
    roof["algorithmic_per_launch"] = {"flops": flops, "bytes": send_bytes}

    line = {
        "metric": METRIC, "value": job_tokens_per_s(world, w.tokens, step_ms), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "e4m3",
        "data": "synthetic (seeded; shapes and laws of the named workload)",
        "config": config_dict(w, q, m_rows, args, world),
        "tflops": tflops,
        "kernels_ms": ({"ep_dispatch_gather": stage_ms[0],
                        "up/gate grouped_gemm_combine_send (local buffer)": stage_ms[1],
                        "ep_swiglu": stage_ms[2], "grouped_gemm_combine_send": stage_ms[3],
                        "ep_combine_reduce": statistics.mean(comb_ms)} if layer else
                       {"grouped_gemm_combine_send (local C)": statistics.mean(gemm_ms),
                        "ep_scatter_send": statistics.mean(send_ms) - statistics.mean(gemm_ms),
                        "ep_combine_reduce": statistics.mean(comb_ms)} if unfused else
                       {"grouped_gemm_combine_send": statistics.mean(send_ms),
                        "ep_combine_reduce": statistics.mean(comb_ms)}),
        "combine_gbs": comb_bytes / comb_s / 1e9,
        "roofline": roof,
        # dispatch, up/gate GEMM (+ ep_swiglu when separate), send, combine; with overlap
        # the serialised copy of every step runs inside the timed loop as well
        "gpu_launches": ((4 if args.layer_act == "fused" else 5) if layer
                         else 3 if unfused else 2) * args.steps * (2 if overlap else 1),
        "clocks": clk,
    }
    if clk and clk.get("sm_mhz"):
        # the dominant kernel's time in SM clock cycles (thousands) at the median clock
        clk["fused_kcycles_at_median_clock"] = dom_s * 1e3 * clk["sm_mhz"]
    if e2e is not None:
        line["e2e"] = e2e
    if args.solo:
        line["config"]["solo"] = "profiling aid: fused send only, peers not staged"
    if layer:
        line["config"]["l2"] = (FLUSH_TEXT if need_flush
                                else f"per-step inputs {step_bytes / 1e6:.0f} MB > L2")
        line["config"]["layer"] = {"hidden": w.N, "intermediate": w.K,
                                   "activation": args.layer_act,
                                   "metric": "tokens/s of the whole layer for one rank"}
    if (rank == 0 and world == 1 and not args.no_per_workload and not args.solo
            and args.path == "fused" and not overlap and args.signal_mode == "rank_flag"
            and args.tokens is None and args.send_warps == -1):
        # every workload's fused send and combine (rank 0 and the most-loaded rank),
        # measured in this process after the headline
        del s, C_local
        torch.cuda.empty_cache()
        pw = {}
        for name in WORKLOADS:
            pw[name] = measure_workload(name, args.pw_steps, max(3, min(args.warmup, 5)),
                                        peaks, peak_src, torch.cuda.current_device())
        line["per_workload"] = pw
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.solo and not layer:
        import oracle
        plans = {r: oracle.plan(w.n_ranks, w.n_local_experts, w.top_k, routing.topk_ids, r)
                 for r in range(w.n_ranks)}
        v, cores, desc, n, dt = cpu_sample(w, routing, values, q, args.cpu_seconds, plans)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
