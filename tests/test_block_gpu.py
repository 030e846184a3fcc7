"""Fused MoE block (RMSNorm -> routed + shared experts -> residual) vs the oracle
(GPU): x_hat and routing bit-exact, outputs to tolerance."""
import numpy as np
import pytest
import torch

from moe_task_scheduling_gb300 import workloads as wl
from tests.helpers import assert_close_bf16
from tests.test_moe_gpu import ODD, SMALL_FINE, SMALL_MIX, WIDE, host_bits

pytestmark = pytest.mark.gpu


def run_block(etmoe, d, b, cfg, T, T_max=None, ws=None, d_T=None, with_xhat=True, **kw):
    dev = torch.device("cuda")
    T_max = T_max or T
    k = cfg.k
    Fs = 0 if b["sg"] is None else b["sg"].shape[0]
    if ws is None:
        ws = etmoe.alloc_workspace(
            etmoe.et_moe_block_workspace_bytes(T_max, cfg.H, cfg.F, cfg.E, k, Fs))
    out = torch.full((T_max, cfg.H), 3.0, dtype=torch.bfloat16, device=dev)
    xhat = torch.full((T_max, cfg.H), 5.0, dtype=torch.bfloat16, device=dev) if with_xhat else None
    idx = torch.full((T_max, k), -1, dtype=torch.int32, device=dev)
    w = torch.full((T_max, k), -1.0, dtype=torch.float32, device=dev)
    cnt = torch.full((cfg.E,), -1, dtype=torch.int32, device=dev)
    perm = torch.full((T_max * k,), -1, dtype=torch.int32, device=dev)
    etmoe.et_moe_block(d["x"], b["gamma"], b["eps"], d["wr"], d["bias"], d["wg"], d["wu"], d["wd"],
                       b["sg"], b["su"], b["sd"], out, k=k, x_hat=xhat,
                       T=T if d_T is None else 0, d_T=d_T, T_max=T_max, topk_idx=idx, topk_w=w,
                       expert_counts=cnt, perm=perm, workspace=ws, **kw)
    torch.cuda.synchronize()
    code, detail = etmoe.et_status(ws)
    return dict(out=out, xhat=xhat, idx=idx.cpu().numpy(), w=w.cpu().numpy(),
                cnt=cnt.cpu().numpy(), perm=perm.cpu().numpy(), code=code, detail=detail, ws=ws)


def oracle_block(oracle, hb, bb, cfg, T, tokens=None):
    return oracle.moe_block(hb["x"][:T], bb["gamma"], bb["eps"], hb["wr"], hb["bias"], hb["wg"],
                            hb["wu"], hb["wd"], bb["sg"], bb["su"], bb["sd"], k=cfg.k,
                            tokens=tokens)


def check_block(res, ref, T, k, sample=None):
    assert res["code"] == 0, f"device status {res['code']} detail {res['detail']}"
    if res["xhat"] is not None:
        assert np.array_equal(wl.bits(res["xhat"])[:T], ref["xhat"]), "x_hat differs"
    assert np.array_equal(res["idx"][:T], ref["idx"]), "top-k indices differ"
    assert np.array_equal(res["cnt"], ref["cnt"]), "expert counts differ"
    assert np.array_equal(res["perm"][:T * k], ref["perm"]), "permutation differs"
    np.testing.assert_allclose(res["w"][:T], ref["w"], rtol=2e-6, atol=1e-7)
    got = wl.bits(res["out"])
    rows = slice(0, T) if sample is None else sample
    assert_close_bf16(got[rows], ref["out"], f"block out T={T}")
    assert torch.all(res["out"][T:].float() == 3.0), "rows >= T must stay untouched"


def _inputs(cfg, Fs, unit, device="cpu"):
    inp = wl.moe_inputs(cfg, device=device, unit_scale=unit)
    blk = wl.block_extra_inputs(cfg, Fs, device=device, unit_scale=unit)
    return inp, blk


def block_bits(blk):
    return {k: (wl.bits(v) if isinstance(v, torch.Tensor) else v) for k, v in blk.items()}


def _to_dev(t):
    return None if t is None else (t.cuda() if isinstance(t, torch.Tensor) else t)


# (config, shared-expert width): no shared expert; one narrower and one wider
# than the routed experts (the wider one splits its down projection over F).
CASES = [(SMALL_MIX, 0), (SMALL_MIX, 1024), (SMALL_FINE, 512), (ODD, 128), (WIDE, 384)]


@pytest.mark.parametrize("cfg,Fs", CASES, ids=lambda c: getattr(c, "name", str(c)))
@pytest.mark.parametrize("unit", [True, False])
def test_block_small_shapes(cuda_lib, oracle, cfg, Fs, unit):
    inp, blk = _inputs(cfg, Fs, unit)
    hb, bb = host_bits(inp), block_bits(blk)
    d = {k: _to_dev(v) for k, v in inp.items()}
    b = {k: _to_dev(v) for k, v in blk.items()}
    for T in cfg.T_sweep:
        res = run_block(cuda_lib, d, b, cfg, T)
        check_block(res, oracle_block(oracle, hb, bb, cfg, T), T, cfg.k)


def test_block_workspace_x_hat(cuda_lib, oracle):
    """x_hat kept in the workspace (no caller buffer): same result."""
    cfg, Fs = SMALL_MIX, 256
    inp, blk = _inputs(cfg, Fs, True)
    hb, bb = host_bits(inp), block_bits(blk)
    d = {k: _to_dev(v) for k, v in inp.items()}
    b = {k: _to_dev(v) for k, v in blk.items()}
    res = run_block(cuda_lib, d, b, cfg, 77, with_xhat=False)
    check_block(res, oracle_block(oracle, hb, bb, cfg, 77), 77, cfg.k)


def test_block_symbolic_T_one_workspace(cuda_lib, oracle):
    """T from device memory over one workspace; every counter back to zero."""
    cfg, Fs = SMALL_MIX, 1024
    T_max = 300
    inp = wl.moe_inputs(cfg, device="cpu", T_max=T_max, unit_scale=True)
    blk = wl.block_extra_inputs(cfg, Fs, unit_scale=True)
    hb, bb = host_bits(inp), block_bits(blk)
    d = {k: _to_dev(v) for k, v in inp.items()}
    b = {k: _to_dev(v) for k, v in blk.items()}
    ws = cuda_lib.alloc_workspace(
        cuda_lib.et_moe_block_workspace_bytes(T_max, cfg.H, cfg.F, cfg.E, cfg.k, Fs))
    d_T = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T in (5, 300, 0, 1, 257, 64, 5):
        d_T.fill_(T)
        res = run_block(cuda_lib, d, b, cfg, T, T_max=T_max, ws=ws, d_T=d_T)
        assert res["code"] == 0
        if T:
            check_block(res, oracle_block(oracle, hb, bb, cfg, T), T, cfg.k)
        else:
            assert torch.all(res["out"].float() == 3.0)
    hdr = res["ws"][:256].view(torch.int32).cpu().numpy()
    assert np.all(hdr[2:] == 0)


def test_block_zero_experts_is_residual_plus_shared(cuda_lib, oracle):
    """Routed experts with zero weights: out = bf16(x + y_shared), still through
    every task of the block."""
    cfg, Fs = SMALL_MIX, 256
    inp, blk = _inputs(cfg, Fs, True)
    for key in ("wg", "wu", "wd"):
        inp[key] = torch.zeros_like(inp[key])
    hb, bb = host_bits(inp), block_bits(blk)
    d = {k: _to_dev(v) for k, v in inp.items()}
    b = {k: _to_dev(v) for k, v in blk.items()}
    res = run_block(cuda_lib, d, b, cfg, 100)
    check_block(res, oracle_block(oracle, hb, bb, cfg, 100), 100, cfg.k)


def test_block_rejects_bad_shared_width(cuda_lib):
    cfg = SMALL_MIX
    assert cuda_lib.et_moe_block_workspace_bytes(64, cfg.H, cfg.F, cfg.E, cfg.k, 100) == 0
    assert cuda_lib.et_moe_block_workspace_bytes(64, cfg.H, cfg.F, cfg.E, cfg.k, -128) == 0
    assert cuda_lib.et_moe_block_workspace_bytes(64, cfg.H, cfg.F, cfg.E, cfg.k, 0) > 0


@pytest.mark.parametrize("cfg,Fs", [(wl.MIXTRAL, 0), (wl.FINE, 1536)], ids=["mixtral", "fine"])
def test_block_full_size(cuda_lib, oracle, cfg, Fs):
    """The configured shapes as a fused block (the fine-grained one with a
    1536-wide shared expert) at every token count of their sweeps, T from device
    memory; x_hat and routing checked for every token, every output row against
    the oracle."""
    inp, blk = _inputs(cfg, Fs, False, device="cuda")
    hb, bb = host_bits(inp), block_bits(blk)
    ws = cuda_lib.alloc_workspace(
        cuda_lib.et_moe_block_workspace_bytes(cfg.T_max, cfg.H, cfg.F, cfg.E, cfg.k, Fs))
    d_T = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T in cfg.T_sweep:
        d_T.fill_(T)
        res = run_block(cuda_lib, inp, blk, cfg, T, T_max=cfg.T_max, ws=ws, d_T=d_T)
        ref = oracle_block(oracle, hb, bb, cfg, T)
        check_block(res, ref, T, cfg.k)


def test_block_fault_times_out_and_recovers(cuda_lib, oracle):
    """A routed gate/up task that skips its release: the block's waits end in
    ET_ERR_TIMEOUT; the next call on the same workspace is correct."""
    cfg, Fs = SMALL_MIX, 1024
    inp, blk = _inputs(cfg, Fs, True)
    hb, bb = host_bits(inp), block_bits(blk)
    d = {k: _to_dev(v) for k, v in inp.items()}
    b = {k: _to_dev(v) for k, v in blk.items()}
    T = 64
    ws = cuda_lib.alloc_workspace(
        cuda_lib.et_moe_block_workspace_bytes(T, cfg.H, cfg.F, cfg.E, cfg.k, Fs))
    res = run_block(cuda_lib, d, b, cfg, T, ws=ws, timeout_us=20000, fault_mode=1, fault_arg=0)
    assert res["code"] == cuda_lib.ET_ERR_TIMEOUT, (res["code"], res["detail"])
    cuda_lib.et_reset_status(ws)
    res = run_block(cuda_lib, d, b, cfg, T, ws=ws)
    check_block(res, oracle_block(oracle, hb, bb, cfg, T), T, cfg.k)
