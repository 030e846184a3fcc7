"""The per-task trace (et_opts.trace) on the GPU: a traced call computes the
same bits as an untraced one, its records are well formed, and a CTA never
writes past its share of the buffer (nor past the buffer)."""
import numpy as np
import pytest
import torch

from moe_task_scheduling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ROLES = {0, 1, 2, 3, 4, 5, 6}  # producer, workers, CTA set-up, exit, phase marks, fills, acc ready


def _records_ok(recs, grid):
    """Every record: a CTA of the grid, a known role, begin <= end; every CTA
    recorded its set-up (role 2)."""
    assert recs, "no trace record"
    for (ty, role, a, b, cta, t0, t1) in recs:
        assert 0 <= cta < grid, cta
        assert role in ROLES, role
        assert 0 < t0 <= t1, (t0, t1)
    assert {r[4] for r in recs if r[1] == 2} == set(range(grid)), "a CTA without its set-up record"


def _guarded(cap, guard=4096):
    """A trace buffer of `cap` records inside a larger zeroed allocation: the
    view handed to the call, and the guard bytes after it."""
    full = torch.zeros(32 + 32 * cap + guard, dtype=torch.uint8, device="cuda")
    return full[:32 + 32 * cap], full[32 + 32 * cap:]


def _moe_call(etmoe, d, cfg, T, trace=None):
    ws = etmoe.alloc_workspace(etmoe.et_moe_workspace_bytes(T, cfg.H, cfg.F, cfg.E, cfg.k))
    out = torch.full((T, cfg.H), 3.0, dtype=torch.bfloat16, device="cuda")
    cnt = torch.zeros(cfg.E, dtype=torch.int32, device="cuda")
    etmoe.et_moe_layer(d["x"], d["wr"], d["bias"], d["wg"], d["wu"], d["wd"], out, k=cfg.k, T=T,
                       T_max=T, expert_counts=cnt, workspace=ws, trace=trace)
    torch.cuda.synchronize()
    assert etmoe.et_status(ws) == (0, 0)
    return out, cnt


@pytest.mark.parametrize("T", [1, 64, 300])
def test_moe_trace_changes_no_result(cuda_lib, T):
    cfg = wl.MoEConfig("fine_small", 4, H=256, F=256, E=128, k=8, T_sweep=(T,), zipf_s=1.2)
    inp = wl.moe_inputs(cfg, device="cuda", T_max=T)
    ref, ref_cnt = _moe_call(cuda_lib, inp, cfg, T)
    buf = cuda_lib.alloc_trace(200000)
    got, got_cnt = _moe_call(cuda_lib, inp, cfg, T, trace=buf)
    assert torch.equal(got, ref), "a traced call computed different outputs"
    assert torch.equal(got_cnt, ref_cnt)
    recs = cuda_lib.read_trace(buf)
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    _records_ok(recs, grid)
    # every routed expert tile appears as worker tasks; the exit of every CTA is recorded
    assert {r[4] for r in recs if r[1] == 3} == set(range(grid))
    assert any(r[1] == 1 and r[0] == 4 for r in recs), "no gate/up task recorded"
    assert any(r[1] == 1 and r[0] == 5 for r in recs), "no down task recorded"


def test_moe_trace_small_buffer_stays_in_bounds(cuda_lib):
    """Far fewer records than tasks: each CTA keeps to its trace_cap / grid
    records and nothing lands past the buffer."""
    cfg = wl.MoEConfig("fine_small", 4, H=256, F=256, E=128, k=8, T_sweep=(300,), zipf_s=1.2)
    inp = wl.moe_inputs(cfg, device="cuda", T_max=300)
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    cap = 3 * grid + 5  # three records a CTA (the 5 left over belong to no CTA)
    buf, guard = _guarded(cap)
    ref, _ = _moe_call(cuda_lib, inp, cfg, 300)
    got, _ = _moe_call(cuda_lib, inp, cfg, 300, trace=buf)
    assert torch.equal(got, ref)
    assert torch.count_nonzero(guard).item() == 0, "trace records past the buffer"
    raw = buf.cpu().numpy()
    rec = raw[32:].reshape(-1, 32)
    ctas = rec[:, 12:16].copy().view(np.int32).ravel()
    used = np.any(rec != 0, axis=1)
    per = cap // grid
    for i in np.nonzero(used)[0]:
        assert i // per == ctas[i] and i < per * grid, f"record {i} outside CTA {ctas[i]}'s share"


def test_splitk_and_mlp_trace_change_no_result(cuda_lib):
    g = torch.Generator().manual_seed(5)
    X = (torch.randn(40, 2048, generator=g)).to(torch.bfloat16).cuda()
    W = (torch.randn(1024, 2048, generator=g) / 45.0).to(torch.bfloat16).cuda()
    ws = cuda_lib.alloc_workspace(cuda_lib.et_splitk_workspace_bytes(40, 1024, 2048, 4))
    Y0 = torch.zeros(40, 1024, dtype=torch.bfloat16, device="cuda")
    Y1 = torch.zeros_like(Y0)
    cuda_lib.et_splitk_gemm(X, W, Y0, split=4, workspace=ws)
    buf = cuda_lib.alloc_trace(20000)
    cuda_lib.et_splitk_gemm(X, W, Y1, split=4, workspace=ws, trace=buf)
    torch.cuda.synchronize()
    assert cuda_lib.et_status(ws) == (0, 0)
    assert torch.equal(Y0, Y1)
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    _records_ok(cuda_lib.read_trace(buf), grid)

    cfg = wl.MLPConfig("mlp_small", 21, H=512, F=1024, eps=1e-5, B_sweep=(16,))
    d = {k: v.cuda() for k, v in wl.mlp_inputs(cfg, device="cpu").items()}
    wsm = cuda_lib.alloc_workspace(cuda_lib.et_mlp_workspace_bytes(16, 512, 1024))
    outs = []
    for trace in (None, cuda_lib.alloc_trace(20000)):
        out = torch.zeros(16, 512, dtype=torch.bfloat16, device="cuda")
        cuda_lib.et_mlp_chain(d["x"], d["gamma"], cfg.eps, d["wg"], d["wu"], d["wd"], out, B=16,
                              B_max=16, workspace=wsm, trace=trace)
        torch.cuda.synchronize()
        assert cuda_lib.et_status(wsm) == (0, 0)
        outs.append((out, trace))
    assert torch.equal(outs[0][0], outs[1][0])
    _records_ok(cuda_lib.read_trace(outs[1][1]), grid)
