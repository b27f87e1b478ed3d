"""The C-ABI library builds for sm_103a, loads, exports every entry point the
header declares, and rejects bad arguments on the host (no GPU needed: argument
checks run before any CUDA call)."""

import ctypes
import os
import re

import pytest

import moe_expert_gemm_gb300 as ep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_ep.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\([^;{]*\)\s*;", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    ep.build()
    return ep.load()


def test_header_declares_the_entry_points():
    assert set(declared_functions()) >= set(ep.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def _cfg(**kw):
    base = dict(n_ranks=4, my_rank=0, n_local_experts=2, top_k=2, num_tokens=64,
                max_tokens_per_rank=64, K=256, N=128, msg_bytes=256, dtype=ep.EP_BF16,
                send_warps=-1, signal_mode=0)
    base.update(kw)
    return ep.ep_config(**base)


def test_plan_sizes(lib):
    assert ep.ep_plan_sizes(_cfg()) == 64 * 4 * 2
    assert ep.ep_plan_sizes(_cfg(n_local_experts=1, n_ranks=8)) == 64 * 8 * 1


@pytest.mark.parametrize("kw,code", [
    (dict(n_ranks=9, my_rank=0), ep.EP_ERR_UNSUPPORTED),  # reach of direct stores is 8 ranks
    (dict(my_rank=4), ep.EP_ERR_INVALID_ARG),
    (dict(msg_bytes=250), ep.EP_ERR_INVALID_ARG),
    (dict(num_tokens=65), ep.EP_ERR_INVALID_ARG),
    (dict(top_k=9), ep.EP_ERR_INVALID_ARG),
    (dict(n_local_experts=300, top_k=2), ep.EP_ERR_UNSUPPORTED),
    (dict(dtype=7), ep.EP_ERR_INVALID_ARG),
    (dict(send_warps=3), ep.EP_ERR_INVALID_ARG),
    (dict(signal_mode=2), ep.EP_ERR_INVALID_ARG),
])
def test_bad_config_rejected_before_launch(lib, kw, code):
    cfg = _cfg(**kw)
    out = ctypes.c_int64(0)
    assert lib.ep_plan_sizes(ctypes.byref(cfg), ctypes.byref(out)) == code
    args = ep.ep_send_args()
    assert lib.grouped_gemm_combine_send(ctypes.byref(cfg), ctypes.byref(args), None) == code
    cargs = ep.ep_combine_args()
    assert lib.ep_combine_reduce(ctypes.byref(cfg), ctypes.byref(cargs), None) == code


def test_zero_args_are_rejected(lib):
    """Zero-initialised send arguments (every pointer NULL) never launch."""
    cfg = _cfg()
    assert lib.grouped_gemm_combine_send(ctypes.byref(cfg), ctypes.byref(ep.ep_send_args()),
                                         None) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_plan(ctypes.byref(cfg), None, ctypes.byref(ep.ep_plan_out()),
                       None) == ep.EP_ERR_INVALID_ARG


def test_unaligned_operand_rejected(lib):
    cfg = _cfg()
    a = ep.ep_send_args()
    a.A, a.W = 0x1000008, 0x2000000
    a.expert_offsets = a.src_info = a.seg_offsets = a.send_counts = a.status = 0x3000000
    a.max_rows = 8
    for r in range(4):
        a.recv_buf_ptrs[r] = 0x4000000 + r * 0x100000
        a.recv_count_ptrs[r] = 0x5000000 + r * 0x100000
    a.atomic_counter = a.rank_completion_counter = 0x6000000
    assert lib.grouped_gemm_combine_send(ctypes.byref(cfg), ctypes.byref(a), None) == \
        ep.EP_ERR_INVALID_ARG


def test_unaligned_src_info_rejected(lib):
    """src_info is accessed as 8-byte (src_idx, src_topk) pairs."""
    cfg = _cfg()
    out = ep.ep_plan_out(0x1000, 0x2000004, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 64)
    assert lib.ep_plan(ctypes.byref(cfg), ctypes.c_void_p(0x8000), ctypes.byref(out),
                       None) == ep.EP_ERR_INVALID_ARG
    a = ep.ep_send_args()
    a.A, a.W = 0x1000000, 0x2000000
    a.expert_offsets = a.seg_offsets = a.send_counts = a.status = 0x3000000
    a.src_info = 0x3000004
    a.max_rows = 8
    for r in range(4):
        a.recv_buf_ptrs[r] = 0x4000000 + r * 0x100000
        a.recv_count_ptrs[r] = 0x5000000 + r * 0x100000
    a.atomic_counter = a.rank_completion_counter = 0x6000000
    assert lib.grouped_gemm_combine_send(ctypes.byref(cfg), ctypes.byref(a), None) == \
        ep.EP_ERR_INVALID_ARG


def test_scatter_send_rejects_bad_arguments(lib):
    """The unfused send step validates like the fused call, before any launch."""
    cfg = _cfg()
    assert lib.ep_scatter_send(ctypes.byref(cfg), ctypes.byref(ep.ep_scatter_args()),
                               None) == ep.EP_ERR_INVALID_ARG
    a = ep.ep_scatter_args()
    a.C = 0x1000000
    a.expert_offsets = a.seg_offsets = a.send_counts = a.status = 0x3000000
    a.src_info = 0x3000008
    a.block_counter = 0x6000000
    a.max_rows = 8
    for r in range(4):
        a.recv_buf_ptrs[r] = 0x4000000 + r * 0x100000
        a.recv_count_ptrs[r] = 0x5000000 + r * 0x100000
    for field, bad in (("C", 0x1000008), ("src_info", 0x3000004), ("block_counter", 0x6000002)):
        b = ep.ep_scatter_args.from_buffer_copy(a)
        setattr(b, field, bad)
        assert lib.ep_scatter_send(ctypes.byref(cfg), ctypes.byref(b), None) == \
            ep.EP_ERR_INVALID_ARG, field
    b = ep.ep_scatter_args.from_buffer_copy(a)
    b.recv_buf_ptrs[2] = 0
    assert lib.ep_scatter_send(ctypes.byref(cfg), ctypes.byref(b), None) == ep.EP_ERR_INVALID_ARG
    bad_cfg = _cfg(n_ranks=9)
    assert lib.ep_scatter_send(ctypes.byref(bad_cfg), ctypes.byref(a), None) == \
        ep.EP_ERR_UNSUPPORTED


def test_fp8_shape_rules(lib):
    """Blockwise fp8 needs whole 128-wide scale blocks along K and N."""
    a = ep.ep_send_args()
    for kw in (dict(K=192), dict(N=320, msg_bytes=640)):
        cfg = _cfg(dtype=ep.EP_FP8_1D2D, **kw)
        assert lib.grouped_gemm_combine_send(ctypes.byref(cfg), ctypes.byref(a), None) == \
            ep.EP_ERR_UNSUPPORTED


def test_bf16_shape_rules(lib):
    """bf16 needs whole 128-byte K atoms and 64-column output chunks; the activation
    epilogue pairs the halves of 256-column tiles."""
    a = ep.ep_send_args()
    for kw in (dict(K=96), dict(N=96, msg_bytes=192)):
        cfg = _cfg(**kw)
        assert lib.grouped_gemm_combine_send(ctypes.byref(cfg), ctypes.byref(a), None) == \
            ep.EP_ERR_UNSUPPORTED
    act = ep.ep_send_args()
    act.p3_control = -1
    act.local_activation = ep.EP_ACT_SWIGLU
    cfg = _cfg(N=192, msg_bytes=384)
    assert lib.grouped_gemm_combine_send(ctypes.byref(cfg), ctypes.byref(act), None) == \
        ep.EP_ERR_UNSUPPORTED


def test_fp8_has_no_dedicated_send_warps(lib):
    """Dedicated send warps exist in the bf16 kernel only."""
    cfg = _cfg(dtype=ep.EP_FP8_1D2D, send_warps=4)
    assert lib.grouped_gemm_combine_send(ctypes.byref(cfg), ctypes.byref(ep.ep_send_args()),
                                         None) == ep.EP_ERR_UNSUPPORTED


def test_per_expert_combine_needs_the_routing(lib):
    """In the per-expert mode the combine waits per token for the token's experts."""
    cfg = _cfg(signal_mode=ep.EP_SIGNAL_PER_EXPERT)
    a = ep.ep_combine_args(0x1000000, 0x2000000, 0x3000000, 0x4000000, 1, 0, 0x5000000, 0, 0)
    assert lib.ep_combine_reduce(ctypes.byref(cfg), ctypes.byref(a), None) == \
        ep.EP_ERR_INVALID_ARG


def test_combine_overlap_mode_is_checked(lib):
    cfg = _cfg()
    a = ep.ep_combine_args(0x1000000, 0x2000000, 0x3000000, 0x4000000, 1, 0, 0x5000000, 0, 3)
    assert lib.ep_combine_reduce(ctypes.byref(cfg), ctypes.byref(a), None) == \
        ep.EP_ERR_INVALID_ARG


def test_ipc_calls_reject_null_arguments(lib):
    h = ep.ep_ipc_handle()
    assert ep.raw_call("ep_ipc_export", None, ctypes.byref(h)) == ep.EP_ERR_INVALID_ARG
    assert ep.raw_call("ep_ipc_import", None, None) == ep.EP_ERR_INVALID_ARG
    assert ep.raw_call("ep_ipc_close", ctypes.byref(h), None) == ep.EP_ERR_INVALID_ARG


def test_strerror(lib):
    assert ep.ep_strerror(ep.EP_ERR_UNSUPPORTED) == "unsupported configuration"
    assert "timed out" in ep.ep_strerror(ep.EP_STATUS_TIMEOUT)


def test_binding_structs_match_the_header(tmp_path):
    """Every argument struct of the binding has the header's size and, field by field,
    its offsets and sizes (a C program built from the header prints them)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = [ep.ep_config, ep.ep_plan_out, ep.ep_send_args, ep.ep_combine_args,
               ep.ep_scatter_args, ep.ep_dispatch_args, ep.ep_swiglu_args, ep.ep_ipc_handle]
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "moe_ep.h"', "int main(void) {"]
    for cls in structs:
        name = cls.__name__
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'printf("{name} {field} %zu %zu\\n", offsetof({name}, {field}), '
                         f'sizeof((({name} *)0)->{field}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    got = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    want = []
    for cls in structs:
        name = cls.__name__
        want.append(f"{name} size {ctypes.sizeof(cls)}")
        for field, _ in cls._fields_:
            d = getattr(cls, field)
            want.append(f"{name} {field} {d.offset} {d.size}")
    assert [g for g in got if g] == want


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "moe_ep.h"

int main(void)
{
    /* the Mixtral-like down-projection of rank 0: 8 ranks x 1 expert, top-2 */
    ep_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.n_ranks = 8; cfg.my_rank = 0; cfg.n_local_experts = 1; cfg.top_k = 2;
    cfg.num_tokens = 4096; cfg.max_tokens_per_rank = 4096; cfg.K = 14336; cfg.N = 4096;
    cfg.msg_bytes = 2 * 4096; cfg.dtype = EP_BF16; cfg.send_warps = -1;
    cfg.signal_mode = EP_SIGNAL_RANK_FLAG;
    int64_t rows = -1;
    int rc = ep_plan_sizes(&cfg, &rows);
    printf("plan_sizes %d %lld\n", rc, (long long)rows);
    cfg.n_ranks = EP_MAX_RANKS + 1;
    printf("too_many_ranks %d\n", ep_plan_sizes(&cfg, &rows));
    ep_ipc_handle h;
    printf("ipc_null %d\n", ep_ipc_export(NULL, &h));
    printf("send_null %d\n", grouped_gemm_combine_send(NULL, NULL, NULL));
    printf("strerror %s\n", ep_strerror(EP_ERR_UNSUPPORTED));
    return 0;
}
"""


def test_a_c_program_links_and_calls_the_library(tmp_path, lib):
    """The boundary from plain C: a program built against include/moe_ep.h and linked
    to libmoe_ep.so calls the host-side entry points (no GPU needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(ep.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lmoe_ep", f"-Wl,-rpath,{libdir}"], check=True,
                   capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = dict(line.split(" ", 1) for line in out if line)
    assert got["plan_sizes"] == f"{ep.EP_OK} {4096 * 8 * 1}"
    assert got["too_many_ranks"] == str(ep.EP_ERR_UNSUPPORTED)
    assert got["ipc_null"] == str(ep.EP_ERR_INVALID_ARG)
    assert got["send_null"] == str(ep.EP_ERR_INVALID_ARG)
    assert got["strerror"] == ep.ep_strerror(ep.EP_ERR_UNSUPPORTED)
