"""Device state of a set of logical EP ranks on one GPU, driven through the C ABI.

PyTorch only allocates device memory and provides streams; every step runs in
``libmoe_ep.so``. On one GPU the receive buffers of the other logical ranks
are separate allocations in the same HBM that stand in for peer memory, so a
producer call for rank r writes into every rank's buffer exactly as it would
over direct peer stores.
"""

from __future__ import annotations

import numpy as np
import torch

from . import (EP_ACT_SWIGLU, EP_BF16, EP_FP8_1D2D, ep_combine_args, ep_combine_reduce, ep_config,
               ep_dispatch_args, ep_dispatch_gather, ep_plan, ep_plan_out, ep_plan_sizes,
               ep_scatter_args, ep_scatter_send, ep_send_args, ep_swiglu, ep_swiglu_args,
               grouped_gemm_combine_send, ptr)

SENTINEL_BYTE = 0xFF  # received bf16 0xFFFF is a NaN: an unwritten slot cannot pass
STATUS_PLAN, STATUS_SEND, STATUS_COMBINE = 0, 1, 2


class EpSystem:
    def __init__(self, n_ranks: int, n_local_experts: int, top_k: int, tokens: int, K: int,
                 N: int, dtype: str = "bf16", device="cuda", max_tokens: int | None = None,
                 timeout_ns: int = 0, send_warps: int = -1, signal_mode: int = 0):
        self.R, self.El, self.k, self.T, self.K, self.N = (n_ranks, n_local_experts, top_k,
                                                           tokens, K, N)
        self.dtype = dtype
        self.dt_code = {"bf16": EP_BF16, "fp8_1d2d": EP_FP8_1D2D}[dtype]
        self.device = torch.device(device)
        self.max_tokens = tokens if max_tokens is None else max_tokens
        self.msg_bytes = 2 * N
        self.timeout_ns = timeout_ns
        self.send_warps = send_warps
        self.signal_mode = signal_mode  # EP_SIGNAL_RANK_FLAG or EP_SIGNAL_PER_EXPERT
        dev = self.device
        R, El = self.R, self.El
        self.recv = [torch.full((self.max_tokens * top_k * self.msg_bytes,), SENTINEL_BYTE,
                                dtype=torch.uint8, device=dev) for _ in range(R)]
        self.counts = [torch.full((El * R + R,), -1, dtype=torch.int64, device=dev)
                       for _ in range(R)]
        self.atomic_counter = [torch.zeros(El, dtype=torch.int32, device=dev) for _ in range(R)]
        self.rank_counter = [torch.zeros(R, dtype=torch.int32, device=dev) for _ in range(R)]
        self.block_counter = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in range(R)]
        self.status = torch.zeros(8, dtype=torch.int32, device=dev)
        self.topk = None
        self.plans: list[dict | None] = [None] * R
        self.ops: list[dict | None] = [None] * R
        self.gates: list[torch.Tensor | None] = [None] * R
        self.out: list[torch.Tensor | None] = [None] * R

    # ------------------------------------------------------------- set-up
    def cfg(self, rank: int) -> ep_config:
        return ep_config(self.R, rank, self.El, self.k, self.T, self.max_tokens, self.K, self.N,
                         self.msg_bytes, self.dt_code, self.send_warps, self.signal_mode)

    def reset_buffers(self):
        for b in self.recv:
            b.fill_(SENTINEL_BYTE)
        for c in self.counts:
            c.fill_(-1)

    def set_routing(self, topk_ids):
        t = torch.as_tensor(np.ascontiguousarray(topk_ids, dtype=np.int32))
        assert tuple(t.shape) == (self.R, self.T, self.k)
        self.topk = t.to(self.device)

    def plan(self, rank: int, stream=None, max_rows: int | None = None) -> dict:
        cap = ep_plan_sizes(self.cfg(rank)) if max_rows is None else max_rows
        dev, El, R = self.device, self.El, self.R
        p = dict(expert_offsets=torch.zeros(El + 1, dtype=torch.int32, device=dev),
                 src_info=torch.zeros((max(cap, 1), 2), dtype=torch.int32, device=dev),
                 seg_offsets=torch.zeros((El, R + 1), dtype=torch.int32, device=dev),
                 send_counts=torch.zeros((El, R), dtype=torch.int32, device=dev),
                 gather_idx=torch.zeros(max(cap, 1), dtype=torch.int32, device=dev),
                 m_total=torch.zeros(1, dtype=torch.int32, device=dev), capacity=cap)
        out = ep_plan_out(ptr(p["expert_offsets"]), ptr(p["src_info"]), ptr(p["seg_offsets"]),
                          ptr(p["send_counts"]), ptr(p["gather_idx"]), ptr(p["m_total"]),
                          self.status.data_ptr() + 4 * STATUS_PLAN, cap)
        ep_plan(self.cfg(rank), self.topk, out, stream)
        self.plans[rank] = p
        return p

    def set_operands(self, rank: int, A: np.ndarray, W: np.ndarray, a_scales=None,
                     w_scales=None, pad_rows: int = 0):
        """Upload a rank's operands (bf16 as uint16 bit patterns, e4m3 as uint8).
        ``pad_rows`` extra rows are appended to A (they are read by tiles that run
        past the last row and never sent)."""
        dev = self.device
        rows = max(A.shape[0] + pad_rows, 1)
        if self.dtype == "bf16":
            a = torch.zeros((rows, self.K), dtype=torch.int16)
            a[:A.shape[0]] = torch.from_numpy(np.ascontiguousarray(A).view(np.int16))
            w = torch.from_numpy(np.ascontiguousarray(W).view(np.int16))
            ops = dict(A=a.view(torch.bfloat16).to(dev), W=w.view(torch.bfloat16).to(dev))
        else:
            a = torch.zeros((rows, self.K), dtype=torch.uint8)
            a[:A.shape[0]] = torch.from_numpy(np.ascontiguousarray(A))
            sa = torch.zeros((rows, self.K // 128), dtype=torch.float32)
            sa[:A.shape[0]] = torch.from_numpy(np.ascontiguousarray(a_scales, dtype=np.float32))
            ops = dict(A=a.to(dev), W=torch.from_numpy(np.ascontiguousarray(W)).to(dev),
                       a_scales=sa.to(dev),
                       w_scales=torch.from_numpy(np.ascontiguousarray(w_scales,
                                                                      dtype=np.float32)).to(dev))
        self.ops[rank] = ops
        return ops

    def set_gates(self, rank: int, gates: np.ndarray):
        self.gates[rank] = torch.from_numpy(np.ascontiguousarray(gates, dtype=np.float32)).to(
            self.device)
        self.out[rank] = torch.zeros((self.T, self.N), dtype=torch.bfloat16, device=self.device)

    # ---------------------------------------------------------------- calls
    def send_args(self, rank: int, epoch: int, p3_control: int = 0, C=None) -> ep_send_args:
        p, o = self.plans[rank], self.ops[rank]
        a = ep_send_args()
        a.A = ptr(o["A"])
        a.a_scales = ptr(o.get("a_scales"))
        a.W = ptr(o["W"])
        a.w_scales = ptr(o.get("w_scales"))
        a.expert_offsets = ptr(p["expert_offsets"])
        a.src_info = ptr(p["src_info"])
        a.seg_offsets = ptr(p["seg_offsets"])
        a.send_counts = ptr(p["send_counts"])
        a.max_rows = min(int(o["A"].shape[0]), int(p["src_info"].shape[0]))
        for d in range(self.R):
            a.recv_buf_ptrs[d] = ptr(self.recv[d])
            a.recv_count_ptrs[d] = ptr(self.counts[d])
        a.atomic_counter = ptr(self.atomic_counter[rank])
        a.rank_completion_counter = ptr(self.rank_counter[rank])
        a.epoch = epoch
        a.p3_control = p3_control
        a.C = ptr(C)
        a.status = self.status.data_ptr() + 4 * STATUS_SEND
        a.trace = None
        a.timeout_ns = self.timeout_ns
        return a

    def send(self, rank: int, epoch: int, stream=None, p3_control: int = 0, C=None,
             overlap: bool = False):
        """``overlap``: may start while the kernel before it on the stream is still
        finishing (programmatic dependent launch; it reads nothing before that kernel
        has completed)."""
        a = self.send_args(rank, epoch, p3_control, C)
        a.overlap_previous = 1 if overlap else 0
        grouped_gemm_combine_send(self.cfg(rank), a, stream)

    def local_C(self, rank: int):
        """A [max_rows][N] bf16 buffer for the unfused path's local GEMM output."""
        return torch.empty((self.ops[rank]["A"].shape[0], self.N), dtype=torch.bfloat16,
                           device=self.device)

    def send_unfused(self, rank: int, epoch: int, C, stream=None):
        """The unfused comparator: the grouped GEMM with the sink disabled stores its
        rows to the local C, then ep_scatter_send moves them and signals."""
        grouped_gemm_combine_send(self.cfg(rank), self.send_args(rank, epoch, -1, C), stream)
        ep_scatter_send(self.cfg(rank), self.scatter_args(rank, epoch, C), stream)

    def scatter_args(self, rank: int, epoch: int, C) -> ep_scatter_args:
        p = self.plans[rank]
        a = ep_scatter_args()
        a.C = ptr(C)
        a.expert_offsets = ptr(p["expert_offsets"])
        a.src_info = ptr(p["src_info"])
        a.seg_offsets = ptr(p["seg_offsets"])
        a.send_counts = ptr(p["send_counts"])
        a.max_rows = min(int(C.shape[0]), int(p["src_info"].shape[0]))
        for d in range(self.R):
            a.recv_buf_ptrs[d] = ptr(self.recv[d])
            a.recv_count_ptrs[d] = ptr(self.counts[d])
        a.block_counter = ptr(self.block_counter[rank])
        a.epoch = epoch
        a.status = self.status.data_ptr() + 4 * STATUS_SEND
        return a

    # ------------------------------------------------------------ whole layer
    def set_layer_operands(self, rank: int, X: np.ndarray, W1: np.ndarray, W2: np.ndarray):
        """Operands of a whole MoE layer around the down-projection (bf16 bit
        patterns): the rank's tokens X [T, H], its experts' up/gate weights W1
        [E_l, 2I, H] (gate rows first) and down-projection weights W2 [E_l, H, I],
        with H = N and I = K. The down-projection's A is produced on the device by
        layer_forward (dispatch, up/gate GEMM, activation)."""
        assert self.dtype == "bf16"
        dev, H, I = self.device, self.N, self.K
        x = torch.zeros((self.max_tokens, H), dtype=torch.int16)
        x[:X.shape[0]] = torch.from_numpy(np.ascontiguousarray(X).view(np.int16))
        rows = max(self.plans[rank]["capacity"], 1)
        self.layer = getattr(self, "layer", [None] * self.R)
        w1 = np.ascontiguousarray(W1).view(np.int16)
        # the same rows in 128-row gate/up blocks, for the activation in the epilogue
        El = w1.shape[0]
        w1i = w1.reshape(El, 2, I // 128, 128, H).transpose(0, 2, 1, 3, 4).reshape(El, 2 * I, H) \
            if I % 128 == 0 else None
        self.layer[rank] = dict(
            X=x.view(torch.bfloat16).to(dev),
            W1=torch.from_numpy(w1).view(torch.bfloat16).to(dev),
            W1i=None if w1i is None else torch.from_numpy(np.ascontiguousarray(w1i)).view(
                torch.bfloat16).to(dev),
            A_in=torch.zeros((rows, H), dtype=torch.bfloat16, device=dev),
            G=torch.zeros((rows, 2 * I), dtype=torch.bfloat16, device=dev))
        self.ops[rank] = dict(
            A=torch.zeros((rows, I), dtype=torch.bfloat16, device=dev),
            W=torch.from_numpy(np.ascontiguousarray(W2).view(np.int16)).view(
                torch.bfloat16).to(dev))

    def cfg_up(self, rank: int) -> ep_config:
        """The up/gate projection's configuration: K = H, N = 2I."""
        return ep_config(self.R, rank, self.El, self.k, self.T, self.max_tokens, self.N,
                         2 * self.K, 4 * self.K, EP_BF16, self.send_warps, self.signal_mode)

    def layer_forward(self, rank: int, epoch: int, stream=None, p3_control: int = 0,
                      events=None, fused_act: bool = False, overlap: bool = False):
        """Dispatch, up/gate GEMM, activation, then the fused down-projection + send
        of producer ``rank`` (every ``layer[r]["X"]`` must hold rank r's tokens).
        ``fused_act``: the activation runs in the up/gate GEMM's epilogue (interleaved
        W1, no G) instead of as its own pass. ``events``: four CUDA events recorded
        after each of the first four steps. ``overlap``: the two GEMM calls launch as
        programmatic dependents of the kernel before them (their set-up overlaps its
        end); ignored when ``events`` are recorded between the steps."""
        L, p = self.layer[rank], self.plans[rank]
        mark = (lambda i: events[i].record(stream)) if events is not None else (lambda i: None)
        d = ep_dispatch_args()
        for r in range(self.R):
            d.x_ptrs[r] = ptr(self.layer[r]["X"])
        d.gather_idx = ptr(p["gather_idx"])
        d.expert_offsets = ptr(p["expert_offsets"])
        d.max_rows = int(L["A_in"].shape[0])
        d.hidden = self.N
        d.A_in = ptr(L["A_in"])
        d.status = self.status.data_ptr() + 4 * STATUS_SEND
        ep_dispatch_gather(self.cfg(rank), d, stream)
        mark(0)
        up = self.send_args(rank, epoch, -1, self.ops[rank]["A"] if fused_act else L["G"])
        up.A = ptr(L["A_in"])
        up.W = ptr(L["W1i"] if fused_act else L["W1"])
        up.max_rows = int(L["A_in"].shape[0])
        if fused_act:
            up.local_activation = EP_ACT_SWIGLU
        overlap = overlap and events is None
        up.overlap_previous = 1 if overlap else 0
        grouped_gemm_combine_send(self.cfg_up(rank), up, stream)
        mark(1)
        if not fused_act:
            a = ep_swiglu_args(ptr(L["G"]), ptr(self.ops[rank]["A"]),
                               ptr(p["expert_offsets"]), int(L["G"].shape[0]), self.K)
            ep_swiglu(self.cfg(rank), a, stream)
        mark(2)
        self.send(rank, epoch, stream, p3_control=p3_control, overlap=overlap)
        mark(3)

    def send_traced(self, rank: int, epoch: int, records: int = 64, stream=None):
        """One send with per-tile timestamps; returns the decoded trace."""
        n_sm = torch.cuda.get_device_properties(self.device).multi_processor_count
        stride = 2 + 4 * records
        buf = torch.zeros(n_sm * stride, dtype=torch.int64, device=self.device)
        a = self.send_args(rank, epoch)
        a.trace = ptr(buf)
        a.trace_records = records
        grouped_gemm_combine_send(self.cfg(rank), a, stream)
        torch.cuda.synchronize()
        return decode_trace(buf.cpu().numpy().view(np.uint64), n_sm, records)

    def combine_args(self, rank: int, epoch: int, gates=None, out=None,
                     overlap: int = 0) -> ep_combine_args:
        g = self.gates[rank] if gates is None else gates
        o = self.out[rank] if out is None else out
        return ep_combine_args(ptr(self.recv[rank]), ptr(self.counts[rank]), ptr(g), ptr(o),
                               epoch, self.timeout_ns,
                               self.status.data_ptr() + 4 * STATUS_COMBINE,
                               ptr(self.topk[rank]) if self.topk is not None else 0,
                               int(overlap))

    def combine(self, rank: int, epoch: int, stream=None, gates=None, out=None,
                overlap: int = 0):
        """``overlap``: EP_OVERLAP_* (True is EP_OVERLAP_ANY): may start while the kernel
        before it on the stream is still finishing (programmatic dependent launch);
        EP_OVERLAP_INPUTS_READY when that kernel writes none of the gates, routing or
        output (e.g. it is the fused send)."""
        ep_combine_reduce(self.cfg(rank), self.combine_args(rank, epoch, gates, out, overlap),
                          stream)

    def publish_peer_flags(self, rank: int, epoch: int):
        """Stand-in for the other ranks finishing on their own GPUs: write the flag
        words of every source rank except ``rank`` in ``rank``'s count buffer."""
        base = self.El * self.R
        idx = [base + q for q in range(self.R) if q != rank]
        if idx:
            self.counts[rank][idx] = epoch

    # -------------------------------------------------------------- readback
    def status_words(self) -> np.ndarray:
        return self.status.cpu().numpy().view(np.uint32)

    def plan_host(self, rank: int) -> dict:
        p = self.plans[rank]
        m = int(p["m_total"].item())
        return dict(expert_offsets=p["expert_offsets"].cpu().numpy(),
                    src_info=p["src_info"][:m].cpu().numpy(),
                    seg_offsets=p["seg_offsets"].cpu().numpy(),
                    send_counts=p["send_counts"].cpu().numpy(),
                    gather_idx=p["gather_idx"][:m].cpu().numpy(), m_total=m)


def decode_trace(words: np.ndarray, n_blocks: int, records: int) -> list:
    """Per thread block: start time and one record per traced tile
    (tile, expert, completed_expert, t_ready, t_stored, t_done), times in ns."""
    stride = 2 + 4 * records
    out = []
    for b in range(n_blocks):
        w = words[b * stride:(b + 1) * stride]
        n = int(w[0])
        recs = []
        for i in range(min(n, records)):
            r = w[2 + 4 * i:6 + 4 * i]
            recs.append(dict(tile=int(r[0] & 0xFFFFFFFF), expert=int((r[0] >> 32) & 0x7FFFFFFF),
                             completed=bool(r[0] >> 63), t_ready=int(r[1]), t_stored=int(r[2]),
                             t_done=int(r[3])))
        out.append(dict(tiles=n, t_start=int(w[1]), records=recs))
    return out


def summarize_trace(tr: list) -> dict:
    """Where a fused launch spends its time, from a decoded trace."""
    starts = [b["t_start"] for b in tr if b["t_start"]]
    recs = [r for b in tr for r in b["records"]]
    if not starts or not recs:
        return {}
    t0 = min(starts)
    t1 = max(r["t_done"] for r in recs)
    epi = [r["t_stored"] - r["t_ready"] for r in recs]
    cnt = [r["t_done"] - r["t_stored"] for r in recs if not r["completed"]]
    sig = [r["t_done"] - r["t_stored"] for r in recs if r["completed"]]
    waits = []
    for b in tr:
        prev = b["t_start"]
        for r in b["records"]:
            waits.append(r["t_ready"] - prev)
            prev = r["t_done"]
    last_end = [max(r["t_done"] for r in b["records"]) - t0 for b in tr if b["records"]]

    def st(x):
        x = np.asarray(x, dtype=np.float64) / 1e3
        return {} if x.size == 0 else dict(n=int(x.size), mean_us=float(x.mean()),
                                           p50_us=float(np.median(x)), max_us=float(x.max()))
    return dict(span_us=(t1 - t0) / 1e3, tiles=len(recs), epilogue=st(epi), count=st(cnt),
                signal=st(sig), wait_for_accumulator=st(waits), block_end=st(last_end))
