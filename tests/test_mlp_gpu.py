"""Statically scheduled MLP chain vs the oracle (GPU)."""
import numpy as np
import pytest
import torch

from moe_task_scheduling_gb300 import workloads as wl
from tests.helpers import assert_close_bf16

pytestmark = pytest.mark.gpu


def run_chain(etmoe, d, eps, B, B_max=None, ws=None, d_B=None, **kw):
    B_max = B_max or B
    H, F = d["x"].shape[1], d["wg"].shape[0]
    if ws is None:
        ws = etmoe.alloc_workspace(etmoe.et_mlp_workspace_bytes(B_max, H, F))
    out = torch.full((B_max, H), 3.0, dtype=torch.bfloat16, device="cuda")
    etmoe.et_mlp_chain(d["x"], d["gamma"], eps, d["wg"], d["wu"], d["wd"], out,
                       B=B if d_B is None else 0, d_B=d_B, B_max=B_max, workspace=ws, **kw)
    torch.cuda.synchronize()
    code, detail = etmoe.et_status(ws)
    return out, code, detail, ws


def small_inputs(B, H, F, seed, unit=True):
    cfg = wl.MLPConfig("mlp_small", seed, H=H, F=F, eps=1e-5, B_sweep=(B,))
    return cfg, wl.mlp_inputs(cfg, device="cpu", unit_scale=unit)


@pytest.mark.parametrize("B,H,F", [(1, 128, 128), (3, 256, 384), (16, 512, 1024), (100, 256, 896),
                                   (256, 384, 256), (300, 256, 512)])
@pytest.mark.parametrize("unit", [True, False])
def test_small_shapes(cuda_lib, oracle, B, H, F, unit):
    cfg, inp = small_inputs(B, H, F, 20 + B, unit)
    hb = {k: wl.bits(v) for k, v in inp.items()}
    d = {k: v.cuda() for k, v in inp.items()}
    out, code, detail, _ = run_chain(cuda_lib, d, cfg.eps, B)
    assert code == 0, (code, detail)
    ref = oracle.mlp_chain(hb["x"], hb["gamma"], cfg.eps, hb["wg"], hb["wu"], hb["wd"])
    assert_close_bf16(wl.bits(out), ref, f"MLP B={B} H={H} F={F}")


def test_symbolic_B(cuda_lib, oracle):
    cfg, inp = small_inputs(64, 256, 512, 40)
    hb = {k: wl.bits(v) for k, v in inp.items()}
    d = {k: v.cuda() for k, v in inp.items()}
    ws = cuda_lib.alloc_workspace(cuda_lib.et_mlp_workspace_bytes(64, 256, 512))
    d_B = torch.zeros(1, dtype=torch.int32, device="cuda")
    for B in (64, 1, 0, 17, 64):
        d_B.fill_(B)
        out, code, detail, _ = run_chain(cuda_lib, d, cfg.eps, B, B_max=64, ws=ws, d_B=d_B)
        assert code == 0, (code, detail)
        assert torch.all(out[B:].float() == 3.0)
        if B:
            ref = oracle.mlp_chain(hb["x"][:B], hb["gamma"], cfg.eps, hb["wg"], hb["wu"], hb["wd"])
            assert_close_bf16(wl.bits(out[:B]), ref, f"MLP B={B}")
    hdr = ws[:256].view(torch.int32).cpu().numpy()
    assert np.all(hdr[2:] == 0)


def test_fault_injection_times_out_cleanly(cuda_lib, oracle):
    cfg, inp = small_inputs(8, 256, 512, 41)
    hb = {k: wl.bits(v) for k, v in inp.items()}
    d = {k: v.cuda() for k, v in inp.items()}
    ws = cuda_lib.alloc_workspace(cuda_lib.et_mlp_workspace_bytes(8, 256, 512))
    out, code, detail, _ = run_chain(cuda_lib, d, cfg.eps, 8, ws=ws, timeout_us=20000,
                                     fault_mode=1, fault_arg=0)
    assert code == cuda_lib.ET_ERR_TIMEOUT, (code, detail)
    cuda_lib.et_reset_status(ws)
    out, code, detail, _ = run_chain(cuda_lib, d, cfg.eps, 8, ws=ws)
    assert code == 0
    ref = oracle.mlp_chain(hb["x"], hb["gamma"], cfg.eps, hb["wg"], hb["wu"], hb["wd"])
    assert_close_bf16(wl.bits(out), ref, "MLP after a timed-out call")


def test_full_size_sweep(cuda_lib, oracle):
    """RMSNorm -> [4096 -> 2x14336] -> SiLU*mul -> [14336 -> 4096], B from device
    memory over every batch size of the configured sweep, every row vs the
    oracle."""
    cfg = wl.MLP
    inp = wl.mlp_inputs(cfg, device="cuda")
    hb = {k: wl.bits(v) for k, v in inp.items()}
    ws = cuda_lib.alloc_workspace(cuda_lib.et_mlp_workspace_bytes(cfg.B_max, cfg.H, cfg.F))
    d_B = torch.zeros(1, dtype=torch.int32, device="cuda")
    for B in cfg.B_sweep:
        d_B.fill_(B)
        out, code, detail, _ = run_chain(cuda_lib, inp, cfg.eps, B, B_max=cfg.B_max, ws=ws, d_B=d_B)
        assert code == 0, (code, detail)
        ref = oracle.mlp_chain(hb["x"][:B], hb["gamma"], cfg.eps, hb["wg"], hb["wu"], hb["wd"])
        assert_close_bf16(wl.bits(out)[:B], ref, f"MLP B={B}")
        assert torch.all(out[B:].float() == 3.0)


def test_ksplit_gate_up_every_row(cuda_lib, oracle):
    """A shape whose gate/up tiles are split along K at small batches (95 F-tiles
    cannot fill the grid): every row against the oracle, one workspace, B read
    from device memory, the counters clean between calls."""
    B_max, H, F = 64, 2048, 95 * 128
    cfg, inp = small_inputs(B_max, H, F, 50)
    hb = {k: wl.bits(v) for k, v in inp.items()}
    d = {k: v.cuda() for k, v in inp.items()}
    ws = cuda_lib.alloc_workspace(cuda_lib.et_mlp_workspace_bytes(B_max, H, F))
    d_B = torch.zeros(1, dtype=torch.int32, device="cuda")
    for B in (1, 17, 64, 33):
        d_B.fill_(B)
        out, code, detail, _ = run_chain(cuda_lib, d, cfg.eps, B, B_max=B_max, ws=ws, d_B=d_B)
        assert code == 0, (code, detail)
        ref = oracle.mlp_chain(hb["x"][:B], hb["gamma"], cfg.eps, hb["wg"], hb["wu"], hb["wd"])
        assert_close_bf16(wl.bits(out)[:B], ref, f"MLP K-split B={B}")
        assert torch.all(out[B:].float() == 3.0)
    hdr = ws[:256].view(torch.int32).cpu().numpy()
    assert np.all(hdr[2:] == 0)
