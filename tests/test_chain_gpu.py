"""Chained MoE layers in one launch (GPU).

- The chain must equal the same layers called one after another, bit for bit
  (the kernel is deterministic for a given shape, token count and grid): a
  layer that read its input before the previous layer had written it would
  differ.
- The first layer is checked against the oracle (routing bit-exact, outputs to
  tolerance), and the whole chain against the oracle applied layer after
  layer: routing on every token whose oracle top-k margin clears a small
  threshold, outputs on the tokens routed alike.
"""
import dataclasses

import numpy as np
import pytest
import torch

from moe_task_scheduling_gb300 import workloads as wl
from tests.helpers import assert_close_bf16
from tests.test_moe_gpu import SMALL_FINE, SMALL_MIX

pytestmark = pytest.mark.gpu


def layer_inputs(cfg, j, block, Fs, unit=True, T_max=None, device="cpu"):
    """Weights of layer j (its own seed); x only matters for layer 0."""
    c = dataclasses.replace(cfg, index=cfg.index + 100 * j)
    inp = wl.moe_inputs(c, device=device, unit_scale=unit, T_max=T_max)
    blk = wl.block_extra_inputs(c, Fs, device=device, unit_scale=unit) if block else None
    return inp, blk


def to_dev(d):
    return None if d is None else {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
                                   for k, v in d.items()}


def bits_of(d):
    return None if d is None else {k: (wl.bits(v) if isinstance(v, torch.Tensor) and
                                       v.dtype == torch.bfloat16 else
                                       (v.cpu().numpy() if isinstance(v, torch.Tensor) else v))
                                   for k, v in d.items()}


class Chain:
    """Device buffers and descriptors of an n-layer chain."""

    def __init__(self, etmoe, cfg, kinds, T_max, unit=True, device="cpu"):
        self.etmoe, self.cfg, self.T_max = etmoe, cfg, T_max
        self.layers = []
        for j, (block, Fs) in enumerate(kinds):
            inp, blk = layer_inputs(cfg, j, block, Fs, unit=unit, T_max=T_max, device=device)
            self.layers.append((to_dev(inp), to_dev(blk), bits_of(inp), bits_of(blk)))
        self.x = self.layers[0][0]["x"]
        dev = torch.device("cuda")
        k, E = cfg.k, cfg.E
        self.outs = [torch.full((T_max, cfg.H), 3.0, dtype=torch.bfloat16, device=dev)
                     for _ in kinds]
        self.idx = [torch.full((T_max, k), -1, dtype=torch.int32, device=dev) for _ in kinds]
        self.cnt = [torch.full((E,), -1, dtype=torch.int32, device=dev) for _ in kinds]

    def descs(self, outs=None, idx=None, cnt=None):
        e = self.etmoe
        outs, idx, cnt = outs or self.outs, idx or self.idx, cnt or self.cnt
        ds = []
        for j, (d, b, _, _) in enumerate(self.layers):
            kw = {} if b is None else dict(gamma=b["gamma"], eps=b["eps"], ws_gate=b["sg"],
                                           ws_up=b["su"], ws_down=b["sd"])
            ds.append(e.layer_desc(d["wr"], d["bias"], d["wg"], d["wu"], d["wd"], outs[j],
                                   topk_idx=idx[j], expert_counts=cnt[j], **kw))
        return ds

    def workspace(self, descs):
        c = self.cfg
        n = self.etmoe.et_moe_chain_workspace_bytes(descs, self.T_max, c.H, c.F, c.E, c.k)
        assert n > 0
        return self.etmoe.alloc_workspace(n)

    def run(self, T, ws=None, d_T=None, x=None):
        """The layers as one chain on input x (default: the chain's x)."""
        c = self.cfg
        descs = self.descs()
        ws = ws if ws is not None else self.workspace(descs)
        self.etmoe.et_moe_chain(descs, self.x if x is None else x, H=c.H, F=c.F, E=c.E, k=c.k,
                                T=T if d_T is None else 0, d_T=d_T, T_max=self.T_max,
                                workspace=ws)
        torch.cuda.synchronize()
        return self.etmoe.et_status(ws)


def oracle_layer(oracle, cfg, x_bits, hb, bb):
    if bb is None:
        r = oracle.moe_layer(x_bits, hb["wr"], hb["bias"], hb["wg"], hb["wu"], hb["wd"], k=cfg.k)
        r["xr"] = x_bits  # the rows the router saw
    else:
        r = oracle.moe_block(x_bits, bb["gamma"], bb["eps"], hb["wr"], hb["bias"], hb["wg"],
                             hb["wu"], hb["wd"], bb["sg"], bb["su"], bb["sd"], k=cfg.k)
        r["xr"] = r["xhat"]
    return r


def topk_margin(oracle, xr_bits, hb, k):
    """Oracle logit gap between the k-th and the (k+1)-th expert, per token."""
    L = oracle.router_logits(xr_bits, hb["wr"], hb["bias"]).astype(np.float64)
    s = -np.sort(-L, axis=1)
    return s[:, k - 1] - s[:, k], L.std()


KINDS = {
    "plain2": [(False, 0), (False, 0)],
    "block2": [(True, 512), (True, 512)],
    "mixed3": [(True, 256), (False, 0), (True, 0)],
    "block4": [(True, 256)] * 4,
}


@pytest.mark.parametrize("kinds", list(KINDS), ids=list(KINDS))
@pytest.mark.parametrize("cfg", [SMALL_MIX, SMALL_FINE], ids=lambda c: c.name)
def test_chain_equals_separate_calls(cuda_lib, cfg, kinds):
    T_max = 300
    ch = Chain(cuda_lib, cfg, KINDS[kinds], T_max)
    ws = ch.workspace(ch.descs())
    d_T = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = len(ch.layers)
    for T in (1, 7, 64, 300, 0, 33):
        d_T.fill_(T)
        for o in ch.outs:
            o.fill_(3.0)
        assert ch.run(T, ws=ws, d_T=d_T) == (0, 0)
        chained = [o.clone() for o in ch.outs]
        idx_c = [i.clone() for i in ch.idx]
        if T == 0:
            assert all(torch.all(o.float() == 3.0) for o in chained)
            continue
        # the same layers, one launch each, each on the previous call's output
        x = ch.x
        for j in range(n):
            for o in ch.outs:
                o.fill_(3.0)
            sub = Chain.__new__(Chain)
            sub.__dict__.update(ch.__dict__)
            sub.layers, sub.outs, sub.idx, sub.cnt = (ch.layers[j:j + 1], ch.outs[j:j + 1],
                                                      ch.idx[j:j + 1], ch.cnt[j:j + 1])
            assert sub.run(T, x=x) == (0, 0)
            assert torch.equal(ch.idx[j][:T], idx_c[j][:T]), f"layer {j} routing, T={T}"
            assert torch.equal(ch.outs[j][:T], chained[j][:T]), f"layer {j} output, T={T}"
            assert torch.all(chained[j][T:].float() == 3.0), "rows >= T must stay untouched"
            x = chained[j]
    # every counter of every layer's region back to zero (headers past the status words)
    hdr = ws[:256].view(torch.int32).cpu().numpy()
    assert np.all(hdr[2:] == 0)


@pytest.mark.parametrize("kinds", ["plain2", "block2"])
def test_chain_vs_oracle(cuda_lib, oracle, kinds):
    cfg = SMALL_MIX
    T = 130
    ch = Chain(cuda_lib, cfg, KINDS[kinds], T)
    assert ch.run(T) == (0, 0)
    x_bits = ch.layers[0][2]["x"][:T]
    checked = 0
    for j, (_, _, hb, bb) in enumerate(ch.layers):
        ref = oracle_layer(oracle, cfg, x_bits, hb, bb)
        got_idx = ch.idx[j][:T].cpu().numpy()
        got_out = wl.bits(ch.outs[j])[:T]
        if j == 0:  # exactly the layer's own parity bar
            assert np.array_equal(got_idx, ref["idx"])
            assert_close_bf16(got_out, ref["out"], "chain layer 0")
        else:
            margin, sd = topk_margin(oracle, ref["xr"], hb, cfg.k)
            # a 1-ulp difference in some input elements moves a logit by ~1e-3 sd
            clear = margin > 2e-2 * sd
            assert clear.mean() > 0.9, "too few tokens with a clear top-k margin"
            same = np.all(np.sort(got_idx, 1) == np.sort(ref["idx"], 1), axis=1)
            assert np.all(same[clear]), f"layer {j}: routing differs on clear tokens"
            assert_close_bf16(got_out[same], ref["out"][same], f"chain layer {j}", rel=2e-2)
            checked += int(same.sum())
        x_bits = ref["out"]  # the oracle chain continues on the oracle's output
    assert checked > 0


def test_chain_mixtral_full_size(cuda_lib, oracle):
    """Two Mixtral-shaped fused blocks (no shared expert) in one launch against
    the two blocks called one after another, T from device memory; every output
    row of the first block against the oracle."""
    cfg = wl.MIXTRAL
    T_max = cfg.T_max
    ch = Chain(cuda_lib, cfg, [(True, 0), (True, 0)], T_max, unit=False, device="cuda")
    ws = ch.workspace(ch.descs())
    d_T = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T in (1, 16, 512):
        d_T.fill_(T)
        assert ch.run(T, ws=ws, d_T=d_T) == (0, 0)
        chained = [o[:T].clone() for o in ch.outs]
        x = ch.x
        for j in range(2):
            sub = Chain.__new__(Chain)
            sub.__dict__.update(ch.__dict__)
            sub.layers, sub.outs, sub.idx, sub.cnt = (ch.layers[j:j + 1], ch.outs[j:j + 1],
                                                      ch.idx[j:j + 1], ch.cnt[j:j + 1])
            assert sub.run(T, x=x) == (0, 0)
            assert torch.equal(ch.outs[j][:T], chained[j]), f"layer {j}, T={T}"
            x = ch.outs[j]
        hb, bb = ch.layers[0][2], ch.layers[0][3]
        ref = oracle.moe_block(hb["x"][:T], bb["gamma"], bb["eps"], hb["wr"], hb["bias"],
                               hb["wg"], hb["wu"], hb["wd"], k=cfg.k)
        assert_close_bf16(wl.bits(chained[0]), ref["out"], f"layer 0 T={T}")


def test_chain_rejects_bad_descriptors(cuda_lib):
    cfg = SMALL_MIX
    ch = Chain(cuda_lib, cfg, KINDS["plain2"], 16)
    ds = ch.descs()
    assert cuda_lib.et_moe_chain_workspace_bytes(ds * 3, 16, cfg.H, cfg.F, cfg.E, cfg.k) == 0
    ds[1].Fs = 128  # a shared expert needs gamma
    assert cuda_lib.et_moe_chain_workspace_bytes(ds, 16, cfg.H, cfg.F, cfg.E, cfg.k) == 0


def test_chain_fault_times_out_and_recovers(cuda_lib):
    """A gate/up task of the first layer that never releases its event: the
    chain must end with ET_ERR_TIMEOUT (every layer unwinds on the launch's
    abort flag), and the next normal call on the same workspace must match
    the same layers launched one by one."""
    cfg = SMALL_MIX
    T = 64
    ch = Chain(cuda_lib, cfg, KINDS["block2"], T)
    descs = ch.descs()
    ws = ch.workspace(descs)
    cuda_lib.et_moe_chain(descs, ch.x, H=cfg.H, F=cfg.F, E=cfg.E, k=cfg.k, T=T, T_max=T,
                          workspace=ws, timeout_us=20000, fault_mode=1, fault_arg=0)
    torch.cuda.synchronize()
    code, detail = cuda_lib.et_status(ws)
    assert code == cuda_lib.ET_ERR_TIMEOUT, (code, detail)
    cuda_lib.et_reset_status(ws)
    for o in ch.outs:
        o.fill_(3.0)
    assert ch.run(T, ws=ws) == (0, 0)
    chained = [o.clone() for o in ch.outs]
    x = ch.x
    for j in range(2):
        sub = Chain.__new__(Chain)
        sub.__dict__.update(ch.__dict__)
        sub.layers, sub.outs, sub.idx, sub.cnt = (ch.layers[j:j + 1], ch.outs[j:j + 1],
                                                  ch.idx[j:j + 1], ch.cnt[j:j + 1])
        assert sub.run(T, x=x) == (0, 0)
        assert torch.equal(ch.outs[j][:T], chained[j][:T]), f"layer {j} after the fault"
        x = chained[j]
