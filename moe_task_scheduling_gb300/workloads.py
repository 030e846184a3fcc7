"""Synthetic workloads: the five layer configurations and their seeded inputs.

This module only draws random inputs with the shapes, scales and structure of
the Event-Tensor MoE workloads.  It computes nothing that the layer computes:
both the CUDA path and the CPU checker receive the tensors made here.

Configurations (all bf16, drawn ~N(0, 0.02) unless stated):
  tiny       T=16,  H=256,  E=8,   k=2, F=512
  splitk     Y[M,4096] = X[M,14336] W, split 8, M in {1, 8, 64, 256}
  mlp        RMSNorm -> gate/up [4096 -> 2x14336] -> SiLU*mul -> down, B 1..256
  mixtral    H=4096, E=8,   k=2, F=14336, T 1..512
  fine       H=2048, E=128, k=8, F=768,   T 1..4096, router logits get a
             per-expert Zipf(s=1.2) bias so that loads are skewed and some
             experts stay empty at small T.

Seeding: one torch.Generator per configuration, seeded 1000 + index, on the
device the tensors are made on (so a CPU draw and a CUDA draw differ, but each
is reproducible).  The activation block is drawn first at the largest token
count and sliced, so every token count of a sweep sees the same weights.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    index: int
    H: int
    F: int
    E: int
    k: int
    T_sweep: tuple
    zipf_s: Optional[float] = None  # per-expert router bias, None = no bias

    @property
    def T_max(self) -> int:
        return max(self.T_sweep)


@dataclasses.dataclass(frozen=True)
class SplitKConfig:
    name: str
    index: int
    N: int
    K: int
    split: int
    M_sweep: tuple

    @property
    def M_max(self) -> int:
        return max(self.M_sweep)


@dataclasses.dataclass(frozen=True)
class MLPConfig:
    name: str
    index: int
    H: int
    F: int
    eps: float
    B_sweep: tuple

    @property
    def B_max(self) -> int:
        return max(self.B_sweep)


TINY = MoEConfig("tiny", 0, H=256, F=512, E=8, k=2, T_sweep=tuple(range(1, 17)))
SPLITK = SplitKConfig("splitk", 1, N=4096, K=14336, split=8, M_sweep=(1, 8, 64, 256))
MLP = MLPConfig("mlp_chain", 2, H=4096, F=14336, eps=1e-5,
                B_sweep=(1, 2, 4, 8, 16, 32, 64, 128, 256))
MIXTRAL = MoEConfig("mixtral", 3, H=4096, F=14336, E=8, k=2,
                    T_sweep=(1, 2, 4, 8, 16, 32, 64, 128, 256, 512))
FINE = MoEConfig("fine_skewed", 4, H=2048, F=768, E=128, k=8,
                 T_sweep=(1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096),
                 zipf_s=1.2)

CONFIGS = {c.name: c for c in (TINY, SPLITK, MLP, MIXTRAL, FINE)}

WEIGHT_STD = 0.02


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, std, g, device, chunk_rows=None):
    """N(0, std^2) drawn in fp32 then rounded to bf16, drawn in row chunks of the
    leading dimension so that very large weights never need a full fp32 copy."""
    shape = tuple(shape)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    lead = shape[0] if shape else 1
    step = chunk_rows or lead
    for i in range(0, lead, step):
        j = min(lead, i + step)
        blk = torch.randn((j - i,) + shape[1:], generator=g, device=device, dtype=torch.float32)
        out[i:j] = (blk * std).to(torch.bfloat16)
    return out


def zipf_router_bias(E: int, H: int, s: float, g, device, x_std=WEIGHT_STD, w_std=WEIGHT_STD):
    """Per-expert logit bias b_e = sigma_L * ln(E * p_e) with p_e proportional to
    r_e^(-s), r a seeded permutation of 1..E, sigma_L the std of a Gaussian logit
    (sqrt(H) * x_std * w_std).  Hot experts sit ~3.5 sigma above the mean, cold
    ones ~2.3 sigma below for E=128, s=1.2."""
    r = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
    p = r.pow(-s)
    p = p / p.sum()
    sigma = math.sqrt(H) * x_std * w_std
    return (sigma * torch.log(E * p)).to(torch.float32)


def moe_inputs(cfg: MoEConfig, device="cpu", T_max: Optional[int] = None, unit_scale=False,
               identical_experts=False):
    """Seeded MoE layer inputs.  Returns dict x [T_max,H], wr [H,E], bias [E] or None,
    wg/wu [E,F,H], wd [E,H,F] (bf16), on `device`.

    unit_scale: x ~ N(0,1) and each weight ~ N(0, 1/fan_in) instead of N(0, 0.02),
    so that outputs are O(1) and an absolute tolerance floor is not vacuous.
    identical_experts: every expert gets expert 0's weights (a special case in
    which the layer must equal one dense SwiGLU MLP)."""
    T_max = T_max or cfg.T_max
    g = _gen(device, 1000 + cfg.index)
    H, F, E = cfg.H, cfg.F, cfg.E
    xs = 1.0 if unit_scale else WEIGHT_STD
    x = _randn_bf16((T_max, H), xs, g, device)
    wr = _randn_bf16((H, E), 1.0 / math.sqrt(H) if unit_scale else WEIGHT_STD, g, device)
    sh = 1.0 / math.sqrt(H) if unit_scale else WEIGHT_STD
    sf = 1.0 / math.sqrt(F) if unit_scale else WEIGHT_STD
    n_draw = 1 if identical_experts else E
    wg = _randn_bf16((n_draw, F, H), sh, g, device, chunk_rows=1)
    wu = _randn_bf16((n_draw, F, H), sh, g, device, chunk_rows=1)
    wd = _randn_bf16((n_draw, H, F), sf, g, device, chunk_rows=1)
    if identical_experts:
        wg, wu, wd = (w.expand(E, -1, -1).contiguous() for w in (wg, wu, wd))
    bias = None
    if cfg.zipf_s is not None:
        bias = zipf_router_bias(E, H, cfg.zipf_s, g, device,
                                x_std=xs, w_std=(1.0 / math.sqrt(H) if unit_scale else WEIGHT_STD))
    return dict(x=x, wr=wr, bias=bias, wg=wg, wu=wu, wd=wd)


def block_extra_inputs(cfg: MoEConfig, Fs: int, device="cpu", unit_scale=False):
    """The fused MoE block's extra inputs (drawn from their own seed, so the
    layer's inputs are unchanged): gamma [H] = 1 + N(0, 0.02), the shared
    expert sg/su [Fs,H], sd [H,Fs] (None when Fs = 0), eps = 1e-5."""
    g = _gen(device, 2000 + cfg.index)
    H = cfg.H
    gamma = (1.0 + torch.randn((H,), generator=g, device=device) * WEIGHT_STD).to(torch.bfloat16)
    sg = su = sd = None
    if Fs:
        sh = 1.0 / math.sqrt(H) if unit_scale else WEIGHT_STD
        sf = 1.0 / math.sqrt(Fs) if unit_scale else WEIGHT_STD
        sg = _randn_bf16((Fs, H), sh, g, device, chunk_rows=1024)
        su = _randn_bf16((Fs, H), sh, g, device, chunk_rows=1024)
        sd = _randn_bf16((H, Fs), sf, g, device, chunk_rows=512)
    return dict(gamma=gamma, sg=sg, su=su, sd=sd, eps=1e-5)


def block_router_bias(layer_bias, unit_scale=False):
    """The skewed router bias for a fused block, whose router sees x_hat (unit
    RMS, gamma ~ 1) instead of x: the same bias in units of the Gaussian logit
    std of x_hat, i.e. scaled by 1 / x_std (None stays None)."""
    if layer_bias is None:
        return None
    return layer_bias * (1.0 if unit_scale else 1.0 / WEIGHT_STD)


def splitk_inputs(cfg: SplitKConfig, device="cpu", M_max: Optional[int] = None, unit_scale=False):
    """X [M_max,K], Wt [N,K] (the weight stored transposed, K contiguous), bf16."""
    M_max = M_max or cfg.M_max
    g = _gen(device, 1000 + cfg.index)
    X = _randn_bf16((M_max, cfg.K), 1.0 if unit_scale else WEIGHT_STD, g, device)
    Wt = _randn_bf16((cfg.N, cfg.K), 1.0 / math.sqrt(cfg.K) if unit_scale else WEIGHT_STD, g,
                     device, chunk_rows=512)
    return dict(X=X, Wt=Wt)


def mlp_inputs(cfg: MLPConfig, device="cpu", B_max: Optional[int] = None, unit_scale=False):
    """x [B_max,H], gamma [H] = 1 + N(0, 0.02), wg/wu [F,H], wd [H,F], bf16."""
    B_max = B_max or cfg.B_max
    g = _gen(device, 1000 + cfg.index)
    H, F = cfg.H, cfg.F
    x = _randn_bf16((B_max, H), 1.0 if unit_scale else WEIGHT_STD, g, device)
    wg = _randn_bf16((F, H), 1.0 / math.sqrt(H) if unit_scale else WEIGHT_STD, g, device,
                     chunk_rows=1024)
    wu = _randn_bf16((F, H), 1.0 / math.sqrt(H) if unit_scale else WEIGHT_STD, g, device,
                     chunk_rows=1024)
    wd = _randn_bf16((H, F), 1.0 / math.sqrt(F) if unit_scale else WEIGHT_STD, g, device,
                     chunk_rows=512)
    gamma = (1.0 + torch.randn((H,), generator=g, device=device) * WEIGHT_STD).to(torch.bfloat16)
    return dict(x=x, gamma=gamma, wg=wg, wu=wu, wd=wd)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bits of a tensor as a host numpy uint16 array (no arithmetic)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """Inverse of bits(): a bf16 tensor holding the given raw bits."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)


def host_f32(a: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    return None if a is None else a.detach().float().cpu().numpy()
