"""The trace buffer's layout as the binding decodes it (CPU): a 32-byte header,
then 32-byte records {int32 type | role << 8, a, b, cta; uint64 t_begin,
t_end}; zero records (t_end == 0) are unused slots."""
import numpy as np
import torch

from moe_task_scheduling_gb300 import etmoe


def _record(type_, role, a, b, cta, t0, t1):
    ints = np.array([type_ | (role << 8), a, b, cta], dtype=np.int32).view(np.uint8)
    ts = np.array([t0, t1], dtype=np.uint64).view(np.uint8)
    return np.concatenate([ints, ts])


def test_read_trace_decodes_records_and_skips_empty_slots():
    cap = 6
    raw = np.zeros(32 + 32 * cap, dtype=np.uint8)
    recs = [(4, 1, 7, 0, 3, 1000, 2500), (17, 4, 12345, 0, 151, 10, 10), (5, 5, -1, 9, 0, 5, 9)]
    for slot, r in zip((0, 2, 5), recs):
        raw[32 + 32 * slot:32 + 32 * (slot + 1)] = _record(*r)
    got = etmoe.read_trace(torch.from_numpy(raw))
    assert got == recs


def test_alloc_trace_capacity_matches_the_options():
    buf = etmoe.alloc_trace(100, device="cpu")
    assert buf.numel() == 32 + 32 * 100 and int(buf.sum()) == 0
    assert etmoe.read_trace(buf) == []
