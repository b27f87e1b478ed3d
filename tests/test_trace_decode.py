"""Host decoding of the fused kernels' per-tile trace records (the layout the header
documents for ep_send_args.trace): per thread block [tiles, start time] then four words
per tile {tile | expert << 32 | completed << 63, ready, stored, done}."""

import numpy as np

from moe_expert_gemm_gb300.system import decode_trace, summarize_trace


def _words(blocks, records):
    stride = 2 + 4 * records
    w = np.zeros(len(blocks) * stride, dtype=np.uint64)
    for b, (start, recs) in enumerate(blocks):
        w[b * stride] = len(recs)
        w[b * stride + 1] = start
        for i, (tile, expert, done, t) in enumerate(recs[:records]):
            base = b * stride + 2 + 4 * i
            w[base] = np.uint64(tile) | (np.uint64(expert) << np.uint64(32)) | \
                (np.uint64(1 << 63) if done else np.uint64(0))
            w[base + 1:base + 4] = t
    return w


def test_records_decode_field_by_field():
    blocks = [(1000, [(7, 3, False, (2000, 2500, 2600)), (159, 255, True, (4000, 4300, 9000))]),
              (1100, [])]
    tr = decode_trace(_words(blocks, 4), 2, 4)
    assert tr[0]["tiles"] == 2 and tr[0]["t_start"] == 1000 and tr[1]["records"] == []
    r0, r1 = tr[0]["records"]
    assert (r0["tile"], r0["expert"], r0["completed"]) == (7, 3, False)
    assert (r1["tile"], r1["expert"], r1["completed"]) == (159, 255, True)
    assert (r1["t_ready"], r1["t_stored"], r1["t_done"]) == (4000, 4300, 9000)


def test_more_tiles_than_records_keeps_the_first():
    blocks = [(0, [(i, 0, False, (10 * i + 1, 10 * i + 2, 10 * i + 3)) for i in range(5)])]
    tr = decode_trace(_words(blocks, 3), 1, 3)
    assert tr[0]["tiles"] == 5 and [r["tile"] for r in tr[0]["records"]] == [0, 1, 2]


def test_summary_spans_and_splits():
    blocks = [(1000, [(0, 0, False, (3000, 4000, 5000)), (1, 0, True, (9000, 10000, 16000))])]
    sm = summarize_trace(decode_trace(_words(blocks, 2), 1, 2))
    assert sm["span_us"] == 15.0 and sm["tiles"] == 2
    assert sm["epilogue"]["mean_us"] == 1.0
    assert sm["count"]["n"] == 1 and sm["count"]["mean_us"] == 1.0
    assert sm["signal"]["n"] == 1 and sm["signal"]["mean_us"] == 6.0
    assert sm["wait_for_accumulator"]["max_us"] == 4.0  # 9000 - 5000
