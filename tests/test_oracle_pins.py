"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test ties one oracle function to something it does not compute itself:
hand-derived goldens, brute force, closed forms, invariants, or a library
routine (numpy/torch) used as an independent check.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from moe_task_scheduling_gb300 import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits_of(vals):
    return wl.bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


def to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------- bf16 rounding

def test_f32_to_bf16_matches_torch(oracle):
    rng = np.random.default_rng(0)
    raw = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # force exact ties (low half = 0x8000) on a quarter of the values
    raw[::4] = (raw[::4] & 0xFFFF0000) | 0x8000
    vals = raw.view(np.float32)
    vals = vals[np.isfinite(vals)]
    ref = wl.bits(torch.from_numpy(vals.copy()).to(torch.bfloat16))
    got = np.array([oracle.f32_to_bf16(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def _rne_bf16_exact(d: float) -> float:
    """Round a finite double to bf16 (8 significant bits) with exact rational arithmetic."""
    if d == 0:
        return d
    q = Fraction(d)
    s = -1 if q < 0 else 1
    q = abs(q)
    e = math.floor(math.log2(q))
    if Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    e = max(e, -126)  # bf16 subnormals share float's minimum exponent
    ulp = Fraction(2) ** (e - 7)
    n = q / ulp
    fl = math.floor(n)
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return float(s * fl * ulp)


def test_f64_to_bf16_single_rounding(oracle):
    rng = np.random.default_rng(1)
    vals = list(rng.normal(0, 1, 3000) * 10.0 ** rng.integers(-6, 6, 3000))
    # doubles that sit just above a bf16 halfway point: a double->float->bf16
    # chain would round them to even, a single rounding must round up
    for m in range(128, 256, 7):
        half = (m + 0.5) / 128.0
        vals.append(half + 2.0 ** -40)
        vals.append(-(half + 2.0 ** -40))
        vals.append(half)  # exact tie
    for v in vals:
        got = oracle.bf16_bits_to_f32(np.array([oracle.f64_to_bf16(v)], np.uint16))[0]
        assert float(got) == _rne_bf16_exact(v), v


# --------------------------------------------------------------------- router logits

def test_router_order_golden(oracle):
    g = json.load(open(os.path.join(GOLD, "router_order.json")))
    H = g["H"]
    w = np.zeros(H)
    for h, v in g["w_nonzero"].items():
        w[int(h)] = v
    got = oracle.router_logit_one(bf16_bits_of(np.ones(H)), bf16_bits_of(w))
    assert got == g["expected_logit"]


def test_router_integer_inputs_exact(oracle):
    """Small-integer inputs: every partial sum is an integer below 2^24, so the
    fixed-order fp32 logits must equal the exact integer dot products."""
    rng = np.random.default_rng(2)
    T, H, E = 9, 4096, 8
    xi = rng.integers(-4, 5, size=(T, H))
    wi = rng.integers(-4, 5, size=(H, E))
    L = oracle.router_logits(bf16_bits_of(xi), bf16_bits_of(wi))
    assert np.array_equal(L.astype(np.int64), xi @ wi)


def test_router_gaussian_within_fp32_bound(oracle):
    """Gaussian inputs: |L - exact| <= gamma_n * sum|x*w| with n = H/32 + 5
    additions per path (standard summation error bound)."""
    rng = np.random.default_rng(3)
    T, H, E = 7, 2048, 16
    xb = bf16_bits_of(rng.normal(0, 0.02, (T, H)))
    wb = bf16_bits_of(rng.normal(0, 0.02, (H, E)))
    L = oracle.router_logits(xb, wb).astype(np.float64)
    xd, wd = to_f64(xb), to_f64(wb)
    exact = xd @ wd
    n = H // 32 + 5
    u = 2.0 ** -24
    bound = (n * u / (1 - n * u)) * (np.abs(xd) @ np.abs(wd))
    assert np.all(np.abs(L - exact) <= bound)
    # and the bound is not vacuous: the error is far smaller than the logits
    assert np.max(np.abs(L - exact)) < 1e-4 * np.max(np.abs(exact))


def test_router_bias_is_one_fp32_add(oracle):
    rng = np.random.default_rng(4)
    T, H, E = 5, 256, 8
    xb = bf16_bits_of(rng.normal(0, 1, (T, H)))
    wb = bf16_bits_of(rng.normal(0, 1, (H, E)))
    b = rng.normal(0, 1, E).astype(np.float32)
    L0 = oracle.router_logits(xb, wb)
    L1 = oracle.router_logits(xb, wb, bias=b)
    assert np.array_equal(L1, (L0 + b[None, :]).astype(np.float32))


# --------------------------------------------------------------------- top-k and gate weights

def test_topk_golden_ties(oracle):
    g = json.load(open(os.path.join(GOLD, "topk_ties.json")))
    for c in g["cases"]:
        L = np.array([c["logits"]], dtype=np.float32)
        idx, w = oracle.topk_gate(L, c["k"])
        assert idx[0].tolist() == c["idx"], c["why"]
        np.testing.assert_allclose(w[0], c["w"], rtol=1e-6, atol=0)


def _brute_topk(L, k):
    """The unique k-subset whose every member outranks every non-member."""
    E = len(L)
    key = lambda e: (-float(L[e]), e)  # noqa: E731  (-0.0 == 0.0 as floats)
    found = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(key(a) < key(b) for a in S for b in rest):
            found.append(sorted(S, key=key))
    assert len(found) == 1
    return found[0]


def test_topk_brute_force_tiny(oracle):
    rng = np.random.default_rng(5)
    E = 8
    for k in (1, 2, 3, 8):
        # coarse values force many ties
        L = (rng.integers(-3, 4, size=(200, E)) * 0.5).astype(np.float32)
        L[0] = 0.0
        L[1, ::2] = -0.0
        idx, w = oracle.topk_gate(L, k)
        for t in range(L.shape[0]):
            assert idx[t].tolist() == _brute_topk(L[t], k)


def test_topk_matches_lexsort(oracle):
    rng = np.random.default_rng(6)
    T, E, k = 500, 128, 8
    L = rng.normal(0, 1, (T, E)).astype(np.float32)
    L[:, 5] = L[:, 77]  # ties between experts 5 and 77
    idx, _ = oracle.topk_gate(L, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -L[t].astype(np.float64)))
        assert idx[t].tolist() == order[:k].tolist()


def test_gate_weights_properties(oracle):
    rng = np.random.default_rng(7)
    L = rng.normal(0, 3, (300, 16)).astype(np.float32)
    idx, w = oracle.topk_gate(L, 4)
    np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, rtol=0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)  # slot order is descending logit
    idx2, w2 = oracle.topk_gate(L, 2)
    L0 = L[np.arange(300), idx2[:, 0]].astype(np.float64)
    L1 = L[np.arange(300), idx2[:, 1]].astype(np.float64)
    np.testing.assert_allclose(w2[:, 0], 1.0 / (1.0 + np.exp(L1 - L0)), rtol=1e-6)
    _, w1 = oracle.topk_gate(L, 1)
    assert np.all(w1 == 1.0)
    # softmax over all experts then top-k then renormalise gives the same weights
    p = np.exp(L.astype(np.float64) - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    sel = np.take_along_axis(p, idx.astype(np.int64), 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-6)


# --------------------------------------------------------------------- dispatch

def test_dispatch_invariants(oracle):
    rng = np.random.default_rng(8)
    for T, E, k in ((1, 8, 2), (37, 8, 2), (300, 128, 8), (64, 4, 4)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        cnt, off, perm, pos = oracle.dispatch(idx, E)
        assert cnt.sum() == T * k
        assert np.array_equal(cnt, np.bincount(idx.ravel(), minlength=E))
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(cnt)]))
        assert np.array_equal(np.sort(perm), np.arange(T * k))  # bijection
        assert np.array_equal(perm[pos], np.arange(T * k))
        flat = idx.ravel()
        for e in range(E):
            seg = perm[off[e]:off[e + 1]]
            assert np.all(flat[seg] == e)
            assert np.all(np.diff(seg // k) > 0)  # ascending tokens, stable


def test_dispatch_all_tokens_same_experts(oracle):
    T, E, k = 10, 8, 2
    idx = np.tile(np.array([[3, 6]], np.int32), (T, 1))
    cnt, off, perm, pos = oracle.dispatch(idx, E)
    assert cnt.tolist() == [0, 0, 0, T, 0, 0, T, 0]
    assert perm[off[3]:off[4]].tolist() == [t * k for t in range(T)]


# --------------------------------------------------------------------- expert FFN and the layer

def _torch_swiglu_f64(xb, wgb, wub, wdb):
    x = torch.from_numpy(to_f64(xb))
    g = x @ torch.from_numpy(to_f64(wgb)).T
    u = x @ torch.from_numpy(to_f64(wub)).T
    h = (torch.nn.functional.silu(g) * u)
    hb = h.to(torch.float32).to(torch.bfloat16).to(torch.float64)  # 1-ulp slack below
    y = hb @ torch.from_numpy(to_f64(wdb)).T
    return h, y


def test_swiglu_row_vs_torch_f64(oracle):
    rng = np.random.default_rng(9)
    H, F = 128, 96
    xb = bf16_bits_of(rng.normal(0, 1, H))
    wg = bf16_bits_of(rng.normal(0, 1 / math.sqrt(H), (F, H)))
    wu = bf16_bits_of(rng.normal(0, 1 / math.sqrt(H), (F, H)))
    wd = bf16_bits_of(rng.normal(0, 1 / math.sqrt(F), (H, F)))
    h, y = oracle.swiglu_row(xb, wg, wu, wd)
    h_ref, y_ref = _torch_swiglu_f64(xb[None], wg, wu, wd)
    np.testing.assert_allclose(to_f64(h), h_ref[0].numpy(), rtol=2.0 ** -8, atol=1e-30)
    np.testing.assert_allclose(to_f64(y), y_ref[0].numpy(), rtol=2.0 ** -7, atol=1e-6)


def test_layer_single_expert_is_dense_mlp(oracle):
    """E = k = 1: the gate weight is exactly 1, so the layer is the expert FFN."""
    rng = np.random.default_rng(10)
    T, H, F = 6, 64, 128
    x = bf16_bits_of(rng.normal(0, 1, (T, H)))
    wr = bf16_bits_of(rng.normal(0, 1, (H, 1)))
    wg = bf16_bits_of(rng.normal(0, 0.1, (1, F, H)))
    wu = bf16_bits_of(rng.normal(0, 0.1, (1, F, H)))
    wd = bf16_bits_of(rng.normal(0, 0.1, (1, H, F)))
    r = oracle.moe_layer(x, wr, None, wg, wu, wd, k=1)
    assert np.all(r["w"] == 1.0) and np.all(r["idx"] == 0)
    for t in range(T):
        _, y = oracle.swiglu_row(x[t], wg[0], wu[0], wd[0])
        assert np.array_equal(r["out"][t], y)


def test_layer_identical_experts_is_dense_mlp(oracle):
    """All experts equal: gate weights sum to 1, so out = dense SwiGLU(x) up to one
    bf16 rounding of y * (sum of fp32 weights)."""
    cfg = wl.TINY
    inp = wl.moe_inputs(cfg, unit_scale=True, identical_experts=True)
    x, wr = wl.bits(inp["x"]), wl.bits(inp["wr"])
    wg, wu, wd = wl.bits(inp["wg"]), wl.bits(inp["wu"]), wl.bits(inp["wd"])
    r = oracle.moe_layer(x, wr, None, wg, wu, wd, k=cfg.k)
    _, y_ref = _torch_swiglu_f64(x, wg[0], wu[0], wd[0])
    np.testing.assert_allclose(to_f64(r["out"]), y_ref.numpy(), rtol=2.0 ** -6, atol=1e-3)
    for t in range(x.shape[0]):
        _, y = oracle.swiglu_row(x[t], wg[0], wu[0], wd[0])
        d = np.abs(to_f64(r["out"][t]) - to_f64(y))
        assert np.all(d <= 2.0 ** -7 * np.abs(to_f64(y)) + 1e-30)


def test_layer_brute_force_tiny(oracle):
    """The whole tiny layer against a direct torch fp64 restatement built on
    library primitives: full softmax, torch.topk on (logit, -index) keys,
    per-token dense expert evaluation."""
    cfg = wl.TINY
    inp = wl.moe_inputs(cfg, unit_scale=True)
    x, wr = wl.bits(inp["x"]), wl.bits(inp["wr"])
    wg, wu, wd = wl.bits(inp["wg"]), wl.bits(inp["wu"]), wl.bits(inp["wd"])
    r = oracle.moe_layer(x, wr, None, wg, wu, wd, k=cfg.k)
    L = oracle.router_logits(x, wr).astype(np.float64)
    T = x.shape[0]
    out_ref = np.zeros((T, cfg.H))
    for t in range(T):
        order = np.lexsort((np.arange(cfg.E), -L[t]))[:cfg.k]
        assert r["idx"][t].tolist() == order.tolist()
        p = np.exp(L[t] - L[t].max())
        p = p / p.sum()
        wsel = p[order] / p[order].sum()
        for j, e in enumerate(order):
            _, y = _torch_swiglu_f64(x[t:t + 1], wg[e], wu[e], wd[e])
            out_ref[t] += wsel[j] * y[0].numpy()
    np.testing.assert_allclose(to_f64(r["out"]), out_ref, rtol=2.0 ** -6, atol=2e-3)


def test_layer_token_subset_equals_full(oracle):
    cfg = wl.TINY
    inp = wl.moe_inputs(cfg)
    args = [wl.bits(inp[n]) for n in ("x", "wr")] + [None] + \
        [wl.bits(inp[n]) for n in ("wg", "wu", "wd")]
    full = oracle.moe_layer(*args, k=cfg.k)
    sub = oracle.moe_layer(*args, k=cfg.k, tokens=[3, 0, 15])
    assert np.array_equal(sub["out"], full["out"][[3, 0, 15]])


# --------------------------------------------------------------------- split-K GEMM

def test_splitk_integer_exact(oracle):
    rng = np.random.default_rng(11)
    M, N, K = 5, 24, 512
    Xi = rng.integers(-1, 2, size=(M, K))
    Wi = rng.integers(-1, 2, size=(N, K))
    Y = oracle.splitk_gemm(bf16_bits_of(Xi), bf16_bits_of(Wi), split=8)
    ref = wl.bits(torch.from_numpy((Xi @ Wi.T).astype(np.float32)).to(torch.bfloat16))
    assert np.array_equal(Y, ref)


def test_splitk_split_invariance_and_zero(oracle):
    rng = np.random.default_rng(12)
    M, N, K = 3, 40, 1024
    Xb = bf16_bits_of(rng.normal(0, 1, (M, K)))
    Wb = bf16_bits_of(rng.normal(0, 1 / 32, (N, K)))
    Y1 = to_f64(oracle.splitk_gemm(Xb, Wb, split=1))
    Y8 = to_f64(oracle.splitk_gemm(Xb, Wb, split=8))
    ref = to_f64(Xb) @ to_f64(Wb).T
    np.testing.assert_allclose(Y1, ref, rtol=2.0 ** -8, atol=0)
    np.testing.assert_allclose(Y8, ref, rtol=2.0 ** -8, atol=0)
    assert np.max(np.abs(Y1 - Y8) / np.abs(ref)) <= 2.0 ** -7
    Z = oracle.splitk_gemm(np.zeros_like(Xb), Wb, split=8)
    assert np.all(to_f64(Z) == 0)
    rows = oracle.splitk_gemm(Xb, Wb, split=8, rows=[2, 0])
    assert np.array_equal(rows, oracle.splitk_gemm(Xb, Wb, split=8)[[2, 0]])


# --------------------------------------------------------------------- RMSNorm and the MLP chain

def test_rmsnorm_constant_row_closed_form(oracle):
    H, eps = 4096, 1e-5
    rng = np.random.default_rng(13)
    gamma_b = bf16_bits_of(1.0 + rng.normal(0, 0.02, H))
    for c in (0.5, -3.0, 0.015625, 1e-3):
        xb = bf16_bits_of(np.full(H, c))
        cb = float(to_f64(xb)[0])
        got = to_f64(oracle.rmsnorm_row(xb, gamma_b, eps))
        ref = math.copysign(1.0, cb) * to_f64(gamma_b) / math.sqrt(1.0 + eps / (cb * cb))
        np.testing.assert_allclose(got, ref, rtol=2.0 ** -8, atol=0)


def test_rmsnorm_scale_invariance(oracle):
    rng = np.random.default_rng(14)
    H = 1024
    g = bf16_bits_of(np.ones(H))
    xb = bf16_bits_of(rng.normal(0, 1, H))
    x2 = bf16_bits_of(to_f64(xb) * 4.0)  # exact power-of-two scaling
    a = oracle.rmsnorm_row(xb, g, 0.0)
    b = oracle.rmsnorm_row(x2, g, 0.0)
    assert np.array_equal(a, b)
    ms = np.mean(to_f64(oracle.rmsnorm_row(xb, g, 0.0)) ** 2)
    assert abs(ms - 1.0) < 1e-2


def test_mlp_chain_is_norm_then_single_expert(oracle):
    rng = np.random.default_rng(15)
    B, H, F = 4, 128, 256
    x = bf16_bits_of(rng.normal(0, 1, (B, H)))
    gamma = bf16_bits_of(1.0 + rng.normal(0, 0.02, H))
    wg = bf16_bits_of(rng.normal(0, 1 / math.sqrt(H), (F, H)))
    wu = bf16_bits_of(rng.normal(0, 1 / math.sqrt(H), (F, H)))
    wd = bf16_bits_of(rng.normal(0, 1 / math.sqrt(F), (H, F)))
    out = oracle.mlp_chain(x, gamma, 1e-5, wg, wu, wd)
    for b in range(B):
        xh = oracle.rmsnorm_row(x[b], gamma, 1e-5)
        _, y = oracle.swiglu_row(xh, wg, wu, wd)
        assert np.array_equal(out[b], y)
    # and against torch fp64: RMSNorm by torch ops, then the SwiGLU FFN
    xd = torch.from_numpy(to_f64(x))
    xn = xd * torch.rsqrt((xd * xd).mean(1, keepdim=True) + 1e-5) * torch.from_numpy(to_f64(gamma))
    xnb = wl.bits(xn.to(torch.float32).to(torch.bfloat16))
    _, y_ref = _torch_swiglu_f64(xnb, wg, wu, wd)
    np.testing.assert_allclose(to_f64(out), y_ref.numpy(), rtol=2.0 ** -5, atol=2e-2)


# --------------------------------------------------------------------- the fused MoE block (R14)

def _block_case(unit, Fs=96, seed_cfg=wl.TINY):
    inp = wl.moe_inputs(seed_cfg, unit_scale=unit)
    ex = wl.block_extra_inputs(seed_cfg, Fs, unit_scale=unit)
    b = {k: wl.bits(v) for k, v in inp.items() if v is not None and v.dtype == torch.bfloat16}
    b.update({k: wl.bits(v) for k, v in ex.items() if isinstance(v, torch.Tensor)})
    return b, ex["eps"], seed_cfg


def test_block_zero_weights_is_residual(oracle):
    """Every expert weight zero (routed and shared): out = x exactly."""
    b, eps, cfg = _block_case(True)
    z = {n: np.zeros_like(b[n]) for n in ("wg", "wu", "wd", "sg", "su", "sd")}
    r = oracle.moe_block(b["x"], b["gamma"], eps, b["wr"], None, z["wg"], z["wu"], z["wd"],
                         z["sg"], z["su"], z["sd"], k=cfg.k)
    assert np.array_equal(r["out"], b["x"])


def test_block_routing_is_layer_routing_of_normed_x(oracle):
    b, eps, cfg = _block_case(True)
    r = oracle.moe_block(b["x"], b["gamma"], eps, b["wr"], None, b["wg"], b["wu"], b["wd"],
                         b["sg"], b["su"], b["sd"], k=cfg.k)
    xh = np.stack([oracle.rmsnorm_row_f32(b["x"][t], b["gamma"], eps)
                   for t in range(b["x"].shape[0])])
    assert np.array_equal(r["xhat"], xh)
    lay = oracle.moe_layer(xh, b["wr"], None, b["wg"], b["wu"], b["wd"], k=cfg.k, want_out=False)
    for n in ("idx", "w", "cnt", "perm"):
        assert np.array_equal(r[n], lay[n]), n


def test_block_shared_only_is_residual_plus_shared_expert(oracle):
    """Routed down weights zero: out = bf16(x + y_s), y_s = the shared SwiGLU of
    x_hat (two bf16 values add exactly in fp64: one rounding, bit-exact)."""
    b, eps, cfg = _block_case(True)
    r = oracle.moe_block(b["x"], b["gamma"], eps, b["wr"], None, b["wg"], b["wu"],
                         np.zeros_like(b["wd"]), b["sg"], b["su"], b["sd"], k=cfg.k)
    ys = np.stack([oracle.swiglu_row(r["xhat"][t], b["sg"], b["su"], b["sd"])[1]
                   for t in range(b["x"].shape[0])])
    ref = np.array([[oracle.f64_to_bf16(a + c) for a, c in zip(xr, yr)]
                    for xr, yr in zip(to_f64(b["x"]), to_f64(ys))], dtype=np.uint16)
    assert np.array_equal(r["out"], ref)


def test_block_vs_torch_f64(oracle):
    """The whole block restated with torch fp64 primitives (RMSNorm, full softmax
    + lexsort top-k on the oracle's fixed-order logits, per-token SwiGLU of the
    routed and the shared expert, residual)."""
    b, eps, cfg = _block_case(True)
    r = oracle.moe_block(b["x"], b["gamma"], eps, b["wr"], None, b["wg"], b["wu"], b["wd"],
                         b["sg"], b["su"], b["sd"], k=cfg.k)
    xd = torch.from_numpy(to_f64(b["x"]))
    xn = xd * torch.rsqrt((xd * xd).mean(1, keepdim=True) + eps) * torch.from_numpy(to_f64(b["gamma"]))
    xnb = wl.bits(xn.to(torch.float32).to(torch.bfloat16))
    L = oracle.router_logits(xnb, b["wr"]).astype(np.float64)
    T = xd.shape[0]
    out_ref = to_f64(b["x"]).copy()
    for t in range(T):
        order = np.lexsort((np.arange(cfg.E), -L[t]))[:cfg.k]
        assert r["idx"][t].tolist() == order.tolist()
        p = np.exp(L[t] - L[t].max())
        wsel = p[order] / p[order].sum()
        for j, e in enumerate(order):
            _, y = _torch_swiglu_f64(xnb[t:t + 1], b["wg"][e], b["wu"][e], b["wd"][e])
            out_ref[t] += wsel[j] * y[0].numpy()
        _, ys = _torch_swiglu_f64(xnb[t:t + 1], b["sg"], b["su"], b["sd"])
        out_ref[t] += ys[0].numpy()
    np.testing.assert_allclose(to_f64(r["out"]), out_ref, rtol=2.0 ** -6, atol=2e-2)


def test_block_token_subset_equals_full(oracle):
    b, eps, cfg = _block_case(False)
    args = (b["x"], b["gamma"], eps, b["wr"], None, b["wg"], b["wu"], b["wd"], b["sg"], b["su"],
            b["sd"])
    full = oracle.moe_block(*args, k=cfg.k)
    sub = oracle.moe_block(*args, k=cfg.k, tokens=[5, 0, 15])
    assert np.array_equal(sub["out"], full["out"][[5, 0, 15]])


def test_block_rmsnorm_f32_sum_is_router_order(oracle):
    """R15's sum of squares uses R1's order: for any row, ss equals the (golden-
    pinned) fixed-order router logit of x against itself, so x_hat must equal
    the formula evaluated from that logit."""
    rng = np.random.default_rng(21)
    H = 512
    for _ in range(5):
        xb = bf16_bits_of(rng.normal(0, 1, H) * np.exp(rng.normal(0, 2, H)))
        gb = bf16_bits_of(1.0 + rng.normal(0, 0.02, H))
        ss = np.float32(oracle.router_logit_one(xb, xb))
        r = np.float32(1.0) / np.sqrt(np.float32(ss / np.float32(H)) + np.float32(1e-5))
        ref = bf16_bits_of(((to_f64(xb).astype(np.float32) * r) * to_f64(gb).astype(np.float32)))
        assert np.array_equal(oracle.rmsnorm_row_f32(xb, gb, 1e-5), ref)


def test_block_rmsnorm_f32_close_to_f64_and_constant_row(oracle):
    rng = np.random.default_rng(22)
    H = 1024
    gb = bf16_bits_of(1.0 + rng.normal(0, 0.02, H))
    for _ in range(5):
        xb = bf16_bits_of(rng.normal(0, 1, H))
        a = to_f64(oracle.rmsnorm_row_f32(xb, gb, 1e-5))
        d = to_f64(oracle.rmsnorm_row(xb, gb, 1e-5))
        assert np.all(np.abs(a - d) <= 2.0 ** -7 * np.abs(d) + 1e-30)
    # constant row c: ss = H c^2 exactly, x_hat = bf16(c / sqrt(c^2 + eps) * gamma)
    c = 0.5
    xb = bf16_bits_of(np.full(H, c))
    got = to_f64(oracle.rmsnorm_row_f32(xb, gb, 1e-5))
    want = c / math.sqrt(c * c + 1e-5) * to_f64(gb)
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want))
