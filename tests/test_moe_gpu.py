"""MoE megakernel vs the oracle (GPU): routing bit-exact, outputs to tolerance."""
import dataclasses

import numpy as np
import pytest
import torch

from moe_task_scheduling_gb300 import workloads as wl
from tests.helpers import assert_close_bf16

pytestmark = pytest.mark.gpu


def run_layer(etmoe, d, cfg, T, T_max=None, ws=None, d_T=None, out=None, **kw):
    """Call the layer on device tensors `d`; returns numpy results."""
    dev = torch.device("cuda")
    T_max = T_max or T
    k = cfg.k
    if ws is None:
        ws = etmoe.alloc_workspace(etmoe.et_moe_workspace_bytes(T_max, cfg.H, cfg.F, cfg.E, k))
    if out is None:
        out = torch.full((T_max, cfg.H), 3.0, dtype=torch.bfloat16, device=dev)
    idx = torch.full((T_max, k), -1, dtype=torch.int32, device=dev)
    w = torch.full((T_max, k), -1.0, dtype=torch.float32, device=dev)
    cnt = torch.full((cfg.E,), -1, dtype=torch.int32, device=dev)
    perm = torch.full((T_max * k,), -1, dtype=torch.int32, device=dev)
    etmoe.et_moe_layer(d["x"], d["wr"], d["bias"], d["wg"], d["wu"], d["wd"], out, k=k,
                       T=T if d_T is None else 0, d_T=d_T, T_max=T_max, topk_idx=idx, topk_w=w,
                       expert_counts=cnt, perm=perm, workspace=ws, **kw)
    torch.cuda.synchronize()
    code, detail = etmoe.et_status(ws)
    return dict(out=out, idx=idx.cpu().numpy(), w=w.cpu().numpy(), cnt=cnt.cpu().numpy(),
                perm=perm.cpu().numpy(), code=code, detail=detail, ws=ws)


def host_bits(inp):
    return {k: (wl.bits(v) if (v is not None and v.dtype == torch.bfloat16) else
                (None if v is None else v.detach().cpu().numpy())) for k, v in inp.items()}


def check(res, ref, T, k, sample=None):
    assert res["code"] == 0, f"device status {res['code']} detail {res['detail']}"
    assert np.array_equal(res["idx"][:T], ref["idx"]), "top-k indices differ"
    assert np.array_equal(res["cnt"], ref["cnt"]), "expert counts differ"
    assert np.array_equal(res["perm"][:T * k], ref["perm"]), "permutation differs"
    np.testing.assert_allclose(res["w"][:T], ref["w"], rtol=2e-6, atol=1e-7)
    got = wl.bits(res["out"])
    if sample is None:
        assert_close_bf16(got[:T], ref["out"], f"out T={T}")
    else:
        assert_close_bf16(got[sample], ref["out"], f"out T={T} (sampled rows)")


def oracle_layer(oracle, hb, cfg, T, tokens=None):
    return oracle.moe_layer(hb["x"][:T], hb["wr"], hb["bias"], hb["wg"], hb["wu"], hb["wd"],
                            k=cfg.k, tokens=tokens)


@pytest.mark.parametrize("unit", [True, False])
def test_tiny_every_token_count(cuda_lib, oracle, unit):
    cfg = wl.TINY
    inp = wl.moe_inputs(cfg, device="cpu", unit_scale=unit)
    hb = host_bits(inp)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    for T in cfg.T_sweep:
        res = run_layer(cuda_lib, d, cfg, T)
        check(res, oracle_layer(oracle, hb, cfg, T), T, cfg.k)


SMALL_MIX = wl.MoEConfig("mixtral_small", 3, H=512, F=384, E=8, k=2, T_sweep=(1, 3, 17, 64, 100, 130))
SMALL_FINE = wl.MoEConfig("fine_small", 4, H=256, F=256, E=128, k=8, T_sweep=(1, 7, 64, 300),
                          zipf_s=1.2)
ODD = wl.MoEConfig("odd_experts", 5, H=128, F=640, E=12, k=3, T_sweep=(1, 2, 31, 77))
# tall expert tiles, no down split: the 256-column (two weight box) down tiles
WIDE = wl.MoEConfig("wide_down", 6, H=512, F=256, E=4, k=2, T_sweep=(300, 520))
# tall expert tiles with few output tiles: 256-column down tiles split in two
# F-chunks, their partials summed by the last arriver
WIDE_SPLIT = wl.MoEConfig("wide_split", 7, H=512, F=512, E=4, k=2, T_sweep=(130, 200, 256))


@pytest.mark.parametrize("cfg", [SMALL_MIX, SMALL_FINE, ODD, WIDE, WIDE_SPLIT],
                         ids=lambda c: c.name)
@pytest.mark.parametrize("unit", [True, False])
def test_small_shapes(cuda_lib, oracle, cfg, unit):
    inp = wl.moe_inputs(cfg, device="cpu", unit_scale=unit)
    hb = host_bits(inp)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    for T in cfg.T_sweep:
        res = run_layer(cuda_lib, d, cfg, T)
        check(res, oracle_layer(oracle, hb, cfg, T), T, cfg.k)


def test_identical_experts(cuda_lib, oracle):
    cfg = SMALL_MIX
    inp = wl.moe_inputs(cfg, device="cpu", unit_scale=True, identical_experts=True)
    hb = host_bits(inp)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    res = run_layer(cuda_lib, d, cfg, 37)
    check(res, oracle_layer(oracle, hb, cfg, 37), 37, cfg.k)


def test_tied_router_goes_to_lowest_experts(cuda_lib, oracle):
    cfg = dataclasses.replace(SMALL_MIX, E=8, k=2)
    inp = wl.moe_inputs(cfg, device="cpu", unit_scale=True)
    inp["wr"] = inp["wr"][:, :1].expand(-1, cfg.E).contiguous()  # every expert scores the same
    hb = host_bits(inp)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    res = run_layer(cuda_lib, d, cfg, 20)
    ref = oracle_layer(oracle, hb, cfg, 20)
    assert np.all(ref["idx"] == np.array([0, 1]))
    check(res, ref, 20, cfg.k)


def test_symbolic_T_one_workspace(cuda_lib, oracle):
    """T read from device memory: one workspace, any count up to T_max, T=0 is a
    no-op, and counters are clean between calls (same result as a fresh call)."""
    cfg = SMALL_MIX
    T_max = 130
    inp = wl.moe_inputs(cfg, device="cpu", T_max=T_max, unit_scale=True)
    hb = host_bits(inp)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    ws = cuda_lib.alloc_workspace(cuda_lib.et_moe_workspace_bytes(T_max, cfg.H, cfg.F, cfg.E, cfg.k))
    d_T = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T in (5, 130, 0, 1, 64, 5):
        d_T.fill_(T)
        res = run_layer(cuda_lib, d, cfg, T, T_max=T_max, ws=ws, d_T=d_T)
        assert res["code"] == 0
        assert torch.all(res["out"][T:].float() == 3.0), "rows >= T must stay untouched"
        if T:
            check(res, oracle_layer(oracle, hb, cfg, T), T, cfg.k)
    # every counter returned to zero: the header (except status) and event arrays
    hdr = res["ws"][:256].view(torch.int32).cpu().numpy()
    assert np.all(hdr[2:] == 0)


def test_device_T_above_max_is_reported(cuda_lib):
    cfg = wl.TINY
    inp = wl.moe_inputs(cfg, device="cpu")
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    d_T = torch.tensor([cfg.T_max + 1], dtype=torch.int32, device="cuda")
    res = run_layer(cuda_lib, d, cfg, cfg.T_max, d_T=d_T)
    assert res["code"] == cuda_lib.ET_ERR_BOUNDS
    assert torch.all(res["out"].float() == 3.0)


def test_fault_injection_times_out_cleanly(cuda_lib, oracle):
    """A gate/up task that never releases its event: the down tasks waiting on it
    must give up within the budget with ET_ERR_TIMEOUT, and the next normal call
    on the same workspace must be correct."""
    cfg = SMALL_MIX
    inp = wl.moe_inputs(cfg, device="cpu", unit_scale=True)
    hb = host_bits(inp)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    ws = cuda_lib.alloc_workspace(cuda_lib.et_moe_workspace_bytes(64, cfg.H, cfg.F, cfg.E, cfg.k))
    res = run_layer(cuda_lib, d, cfg, 64, ws=ws, timeout_us=20000, fault_mode=1, fault_arg=0)
    assert res["code"] == cuda_lib.ET_ERR_TIMEOUT, (res["code"], res["detail"])
    cuda_lib.et_reset_status(ws)
    res = run_layer(cuda_lib, d, cfg, 64, ws=ws)
    check(res, oracle_layer(oracle, hb, cfg, 64), 64, cfg.k)


@pytest.mark.parametrize("cfg", [wl.MIXTRAL, wl.FINE], ids=["mixtral", "fine"])
def test_full_size(cuda_lib, oracle, cfg):
    """The configured shapes at every token count of their sweeps, one workspace,
    T from device memory.  Routing, counts and the permutation are checked
    bit-exactly and every output row against the oracle."""
    inp = wl.moe_inputs(cfg, device="cuda")
    hb = host_bits(inp)
    ws = cuda_lib.alloc_workspace(cuda_lib.et_moe_workspace_bytes(cfg.T_max, cfg.H, cfg.F, cfg.E,
                                                                  cfg.k))
    d_T = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T in cfg.T_sweep:
        d_T.fill_(T)
        res = run_layer(cuda_lib, inp, cfg, T, T_max=cfg.T_max, ws=ws, d_T=d_T)
        ref = oracle_layer(oracle, hb, cfg, T)
        check(res, ref, T, cfg.k)
        assert torch.all(res["out"][T:].float() == 3.0), "rows >= T must stay untouched"
        if cfg is wl.FINE and T == cfg.T_max:
            hot_expert_tiles_compared(ref, T, cfg.k)


def hot_expert_tiles_compared(ref, T, k):
    """The skewed layer's hottest expert holds rows for several 256-row expert
    tiles (tasks of one expert on different CTAs, each tile with its own event
    counters); check() compared every token, so every row of each of those
    tiles was compared with the oracle."""
    hot = int(np.argmax(ref["cnt"]))
    n_tiles = -(-int(ref["cnt"][hot]) // 256)
    assert n_tiles >= 3, f"hottest expert {hot} has only {ref['cnt'][hot]} rows"
    rows = ref["perm"][ref["off"][hot]:ref["off"][hot + 1]] // k
    for g in range(n_tiles):
        toks = rows[g * 256:(g + 1) * 256]
        assert len(toks) > 0 and np.all(toks < T)
