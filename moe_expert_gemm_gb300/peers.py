"""One expert-parallel rank per process, with its peers' receive buffers mapped
through CUDA IPC handles.

Where ``system.EpSystem`` plays every logical rank in one process (the other
ranks' receive buffers are other allocations of the same process), ``EpRank`` is
the state of one rank in a group of processes on one node, as the pages deploy it:
each rank owns its receive buffer and receive-count buffer, exports both
(``ep_ipc_export``), and maps every peer's (``ep_ipc_import``), so that its fused
send stores rows, count words and the rank flag straight into the peers' memory
("ep_signal_completion": direct memory access when the target device is on the same
node; "P3PeerSendConfig": one receive-buffer pointer per rank). The handle bytes
travel over any host channel; ``exchange`` uses a torch.distributed group (gloo).

PyTorch only allocates device memory here; every step runs in ``libmoe_ep.so``.
A process must keep its buffers allocated until every peer has closed its mapping
(``close``), and must not free them while a peer's send may still store into them.
"""

from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import (EP_BF16, EP_FP8_1D2D, ep_combine_args, ep_combine_reduce, ep_config,
               ep_ipc_close, ep_ipc_export, ep_ipc_handle, ep_ipc_import, ep_plan, ep_plan_out,
               ep_plan_sizes, ep_send_args, grouped_gemm_combine_send, ptr)

SENTINEL_BYTE = 0xFF
STATUS_PLAN, STATUS_SEND, STATUS_COMBINE = 0, 1, 2


def handle_bytes(h: ep_ipc_handle) -> bytes:
    """The handle as plain bytes (to send to another process)."""
    return bytes(ctypes.string_at(ctypes.addressof(h), ctypes.sizeof(h)))


def handle_from_bytes(b: bytes) -> ep_ipc_handle:
    if len(b) != ctypes.sizeof(ep_ipc_handle):
        raise ValueError(f"an IPC handle is {ctypes.sizeof(ep_ipc_handle)} bytes, got {len(b)}")
    return ep_ipc_handle.from_buffer_copy(b)


def peer_tables(my_rank: int, own: tuple, gathered: list, import_fn) -> list:
    """Per buffer kind, the address of every rank's buffer as seen by this process:
    its own buffers as they are, every other rank's through ``import_fn`` applied to
    that rank's exported handle bytes. ``own`` holds this rank's addresses, one per
    kind; ``gathered[r]`` the handle bytes rank r exported, one per kind, in the
    same order."""
    if not 0 <= my_rank < len(gathered):
        raise ValueError(f"rank {my_rank} outside a group of {len(gathered)}")
    kinds = len(own)
    if any(len(g) != kinds for g in gathered):
        raise ValueError("every rank must export the same buffer kinds")
    return [[own[k] if r == my_rank else import_fn(gathered[r][k]) for r in range(len(gathered))]
            for k in range(kinds)]


class EpRank:
    """Device state of rank ``my_rank`` of an ``n_ranks`` expert-parallel group whose
    ranks are separate processes; see the module docstring."""

    def __init__(self, n_ranks: int, my_rank: int, n_local_experts: int, top_k: int,
                 tokens: int, K: int, N: int, dtype: str = "bf16", device="cuda",
                 timeout_ns: int = 0, signal_mode: int = 0, max_tokens: int | None = None):
        self.R, self.rank, self.El, self.k, self.T, self.K, self.N = (
            n_ranks, my_rank, n_local_experts, top_k, tokens, K, N)
        self.dtype = dtype
        self.dt_code = {"bf16": EP_BF16, "fp8_1d2d": EP_FP8_1D2D}[dtype]
        self.device = torch.device(device)
        self.max_tokens = tokens if max_tokens is None else max_tokens
        self.msg_bytes = 2 * N
        self.timeout_ns = timeout_ns
        self.signal_mode = signal_mode
        dev = self.device
        # what the peers write: this rank's receive buffer and receive-count buffer
        self.recv = torch.full((self.max_tokens * top_k * self.msg_bytes,), SENTINEL_BYTE,
                               dtype=torch.uint8, device=dev)
        self.counts = torch.full((n_local_experts * n_ranks + n_ranks,), -1, dtype=torch.int64,
                                 device=dev)
        self.atomic_counter = torch.zeros(n_local_experts, dtype=torch.int32, device=dev)
        self.rank_counter = torch.zeros(n_ranks, dtype=torch.int32, device=dev)
        self.status = torch.zeros(4, dtype=torch.int32, device=dev)
        self.recv_ptrs = [0] * n_ranks
        self.count_ptrs = [0] * n_ranks
        self.imported: list = []
        self.topk = self.plan_dev = self.ops = self.gates = self.out = None

    # ------------------------------------------------------------- peers
    def export_handles(self) -> tuple:
        return (handle_bytes(ep_ipc_export(self.recv)), handle_bytes(ep_ipc_export(self.counts)))

    def attach(self, gathered: list):
        """Map every peer's buffers from the handle bytes each rank exported
        (``gathered[r]`` = rank r's ``export_handles()``)."""
        def imp(b):
            h = handle_from_bytes(b)
            p = ep_ipc_import(h)
            self.imported.append((h, p))
            return p
        self.recv_ptrs, self.count_ptrs = peer_tables(
            self.rank, (ptr(self.recv), ptr(self.counts)), gathered, imp)

    def exchange(self, group=None):
        """Export, all-gather the handles over a torch.distributed group whose ranks
        are this group's ranks, and map the peers' buffers."""
        import torch.distributed as dist
        if dist.get_world_size(group) != self.R or dist.get_rank(group) != self.rank:
            raise ValueError("the process group must hold exactly the expert-parallel ranks")
        gathered = [None] * self.R
        dist.all_gather_object(gathered, self.export_handles(), group=group)
        self.attach(gathered)

    def close(self):
        for h, p in self.imported:
            ep_ipc_close(h, p)
        self.imported = []
        self.recv_ptrs = [0] * self.R
        self.count_ptrs = [0] * self.R

    # ------------------------------------------------------------- set-up
    def cfg(self) -> ep_config:
        return ep_config(self.R, self.rank, self.El, self.k, self.T, self.max_tokens, self.K,
                         self.N, self.msg_bytes, self.dt_code, -1, self.signal_mode)

    def reset_buffers(self):
        self.recv.fill_(SENTINEL_BYTE)
        self.counts.fill_(-1)

    def set_routing(self, topk_ids):
        """Every rank's routing [n_ranks][tokens][top_k] (the plan of this rank reads
        all of it; the per-expert combine reads this rank's part)."""
        t = torch.as_tensor(np.ascontiguousarray(topk_ids, dtype=np.int32))
        assert tuple(t.shape) == (self.R, self.T, self.k)
        self.topk = t.to(self.device)

    def plan(self, stream=None) -> dict:
        cap = ep_plan_sizes(self.cfg())
        dev, El, R = self.device, self.El, self.R
        p = dict(expert_offsets=torch.zeros(El + 1, dtype=torch.int32, device=dev),
                 src_info=torch.zeros((max(cap, 1), 2), dtype=torch.int32, device=dev),
                 seg_offsets=torch.zeros((El, R + 1), dtype=torch.int32, device=dev),
                 send_counts=torch.zeros((El, R), dtype=torch.int32, device=dev),
                 gather_idx=torch.zeros(max(cap, 1), dtype=torch.int32, device=dev),
                 m_total=torch.zeros(1, dtype=torch.int32, device=dev))
        out = ep_plan_out(ptr(p["expert_offsets"]), ptr(p["src_info"]), ptr(p["seg_offsets"]),
                          ptr(p["send_counts"]), ptr(p["gather_idx"]), ptr(p["m_total"]),
                          self.status.data_ptr() + 4 * STATUS_PLAN, cap)
        ep_plan(self.cfg(), self.topk, out, stream)
        self.plan_dev = p
        return p

    def set_operands(self, A: np.ndarray, W: np.ndarray, a_scales=None, w_scales=None):
        """This rank's operands (bf16 as uint16 bit patterns, e4m3 as uint8): A in plan
        order, W [E_l, N, K]."""
        dev = self.device
        rows = max(A.shape[0], 1)
        if self.dtype == "bf16":
            a = torch.zeros((rows, self.K), dtype=torch.int16)
            a[:A.shape[0]] = torch.from_numpy(np.ascontiguousarray(A).view(np.int16))
            self.ops = dict(A=a.view(torch.bfloat16).to(dev),
                            W=torch.from_numpy(np.ascontiguousarray(W).view(np.int16)).view(
                                torch.bfloat16).to(dev))
        else:
            a = torch.zeros((rows, self.K), dtype=torch.uint8)
            a[:A.shape[0]] = torch.from_numpy(np.ascontiguousarray(A))
            sa = torch.zeros((rows, self.K // 128), dtype=torch.float32)
            sa[:A.shape[0]] = torch.from_numpy(np.ascontiguousarray(a_scales, dtype=np.float32))
            self.ops = dict(A=a.to(dev), W=torch.from_numpy(np.ascontiguousarray(W)).to(dev),
                            a_scales=sa.to(dev),
                            w_scales=torch.from_numpy(np.ascontiguousarray(
                                w_scales, dtype=np.float32)).to(dev))

    def set_gates(self, gates: np.ndarray):
        self.gates = torch.from_numpy(np.ascontiguousarray(gates, dtype=np.float32)).to(self.device)
        self.out = torch.zeros((self.T, self.N), dtype=torch.bfloat16, device=self.device)

    # ---------------------------------------------------------------- calls
    def send_args(self, epoch: int) -> ep_send_args:
        if not all(self.recv_ptrs) or not all(self.count_ptrs):
            raise RuntimeError("exchange the peers' handles first")
        p, o = self.plan_dev, self.ops
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
            a.recv_buf_ptrs[d] = self.recv_ptrs[d]
            a.recv_count_ptrs[d] = self.count_ptrs[d]
        a.atomic_counter = ptr(self.atomic_counter)
        a.rank_completion_counter = ptr(self.rank_counter)
        a.epoch = epoch
        a.status = self.status.data_ptr() + 4 * STATUS_SEND
        a.timeout_ns = self.timeout_ns
        return a

    def send(self, epoch: int, stream=None):
        """The fused grouped GEMM + combine send of this rank into every rank's buffers."""
        grouped_gemm_combine_send(self.cfg(), self.send_args(epoch), stream)

    def combine(self, epoch: int, stream=None, timeout_ns: int | None = None):
        """The gate-weighted combine of this rank's tokens from its own receive buffer."""
        a = ep_combine_args(ptr(self.recv), ptr(self.counts), ptr(self.gates), ptr(self.out),
                            epoch, self.timeout_ns if timeout_ns is None else timeout_ns,
                            self.status.data_ptr() + 4 * STATUS_COMBINE,
                            ptr(self.topk[self.rank]) if self.topk is not None else 0, 0)
        ep_combine_reduce(self.cfg(), a, stream)

    # -------------------------------------------------------------- readback
    def status_words(self) -> np.ndarray:
        return self.status.cpu().numpy().view(np.uint32)
