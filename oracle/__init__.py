"""CPU oracle of the Event-Tensor MoE hot path (ctypes wrapper over plain C).

TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the bench's
CPU-baseline / reference leg may import this package.  It shares no code with
the CUDA library and never calls it.

bf16 tensors are passed as numpy uint16 arrays holding the raw bf16 bits.
Every function mirrors one definition in etmoe_oracle.c; see that file for the
readings taken where the source pages are silent.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def lib():
    global _lib
    if _lib is None:
        path = build_oracle()
        L = ctypes.CDLL(path)
        L.eto_bf16_to_f32.restype = ctypes.c_float
        L.eto_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.eto_f32_to_bf16.restype = ctypes.c_uint16
        L.eto_f32_to_bf16.argtypes = [ctypes.c_float]
        L.eto_f64_to_bf16.restype = ctypes.c_uint16
        L.eto_f64_to_bf16.argtypes = [ctypes.c_double]
        L.eto_router_logit_one.restype = ctypes.c_float
        L.eto_router_logit_one.argtypes = [_u16p, ctypes.c_int64, _u16p, ctypes.c_int64,
                                           ctypes.c_int, _f32p]
        L.eto_router_logits.restype = None
        L.eto_router_logits.argtypes = [_u16p, _u16p, _f32p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, _f32p, ctypes.c_int]
        L.eto_topk_gate.restype = None
        L.eto_topk_gate.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, _f32p]
        L.eto_dispatch.restype = None
        L.eto_dispatch.argtypes = [_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, _i32p,
                                   _i32p, _i32p]
        L.eto_swiglu_row.restype = None
        L.eto_swiglu_row.argtypes = [_u16p, _u16p, _u16p, _u16p, ctypes.c_int, ctypes.c_int,
                                     _u16p, _u16p]
        L.eto_moe_layer.restype = ctypes.c_int
        L.eto_moe_layer.argtypes = [_u16p, _u16p, _f32p, _u16p, _u16p, _u16p] + \
            [ctypes.c_int] * 5 + [_i32p, ctypes.c_int, _u16p, _i32p, _f32p, _i32p, _i32p, _i32p,
                                  _i32p, ctypes.c_int]
        L.eto_splitk_gemm.restype = ctypes.c_int
        L.eto_splitk_gemm.argtypes = [_u16p, _u16p] + [ctypes.c_int] * 4 + \
            [_i32p, ctypes.c_int, _u16p, ctypes.c_int]
        L.eto_rmsnorm_row.restype = None
        L.eto_rmsnorm_row.argtypes = [_u16p, _u16p, ctypes.c_double, ctypes.c_int, _u16p]
        L.eto_mlp_chain.restype = ctypes.c_int
        L.eto_mlp_chain.argtypes = [_u16p, _u16p, ctypes.c_float, _u16p, _u16p, _u16p,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int,
                                    _u16p, ctypes.c_int]
        L.eto_rmsnorm_row_f32.restype = None
        L.eto_rmsnorm_row_f32.argtypes = [_u16p, _u16p, ctypes.c_float, ctypes.c_int, _u16p]
        L.eto_moe_block.restype = ctypes.c_int
        L.eto_moe_block.argtypes = [_u16p, _u16p, ctypes.c_float, _u16p, _f32p, _u16p, _u16p,
                                    _u16p, _u16p, _u16p, _u16p] + [ctypes.c_int] * 6 + \
            [_i32p, ctypes.c_int, _u16p, _u16p, _i32p, _f32p, _i32p, _i32p, ctypes.c_int]
        _lib = L
    return _lib


def _p(a, typ):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(typ)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"bf16 bits expected as uint16, got {a.dtype}"
    return a


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


# ---- scalar conversions -------------------------------------------------------

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32 (numpy, no rounding involved)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(v: float) -> int:
    return int(lib().eto_f32_to_bf16(float(v)))


def f64_to_bf16(v: float) -> int:
    return int(lib().eto_f64_to_bf16(float(v)))


# ---- the path's steps -----------------------------------------------------------

def router_logits(x, wr, bias=None, nthreads=None):
    """fp32 logits [T,E] in the fixed order (32 strided partials, halving tree)."""
    x, wr = _u16(x), _u16(wr)
    T, H = x.shape
    E = wr.shape[1]
    out = np.empty((T, E), dtype=np.float32)
    b = _f32(bias)
    lib().eto_router_logits(_p(x, _u16p), _p(wr, _u16p), _p(b, _f32p), T, H, E, _p(out, _f32p),
                            nthreads or default_threads())
    return out


def router_logit_one(xv, wv, bias_e=None):
    xv, wv = _u16(xv), _u16(wv)
    b = None if bias_e is None else np.array([bias_e], dtype=np.float32)
    return float(lib().eto_router_logit_one(_p(xv, _u16p), 1, _p(wv, _u16p), 1, xv.shape[0],
                                            _p(b, _f32p)))


def topk_gate(logits, k):
    logits = _f32(logits)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    lib().eto_topk_gate(_p(logits, _f32p), T, E, k, _p(idx, _i32p), _p(w, _f32p))
    return idx, w


def dispatch(idx, E):
    idx = _i32(idx)
    T, k = idx.shape
    cnt = np.empty(E, dtype=np.int32)
    off = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    pos = np.empty(T * k, dtype=np.int32)
    lib().eto_dispatch(_p(idx, _i32p), T, E, k, _p(cnt, _i32p), _p(off, _i32p), _p(perm, _i32p),
                       _p(pos, _i32p))
    return cnt, off, perm, pos


def swiglu_row(xrow, wg, wu, wd):
    """One expert's FFN on one row: returns (h bf16 [F], y bf16 [H])."""
    xrow, wg, wu, wd = _u16(xrow), _u16(wg), _u16(wu), _u16(wd)
    F, H = wg.shape
    h = np.empty(F, dtype=np.uint16)
    y = np.empty(H, dtype=np.uint16)
    lib().eto_swiglu_row(_p(xrow, _u16p), _p(wg, _u16p), _p(wu, _u16p), _p(wd, _u16p), H, F,
                         _p(h, _u16p), _p(y, _u16p))
    return h, y


def moe_layer(x, wr, bias, wg, wu, wd, k, tokens=None, want_out=True, nthreads=None):
    """The whole MoE layer.  Returns a dict with idx, w, cnt, off, perm, pos and
    out (bf16 bits; rows = `tokens` when given, else all tokens)."""
    x, wr, wg, wu, wd = _u16(x), _u16(wr), _u16(wg), _u16(wu), _u16(wd)
    T, H = x.shape
    E, F, _ = wg.shape
    tok = _i32(tokens)
    n_out = (len(tok) if tok is not None else T) if want_out else 0
    out = np.empty((n_out, H), dtype=np.uint16) if want_out else None
    res = dict(idx=np.empty((T, k), np.int32), w=np.empty((T, k), np.float32),
               cnt=np.empty(E, np.int32), off=np.empty(E + 1, np.int32),
               perm=np.empty(T * k, np.int32), pos=np.empty(T * k, np.int32))
    b = _f32(bias)
    rc = lib().eto_moe_layer(
        _p(x, _u16p), _p(wr, _u16p), _p(b, _f32p), _p(wg, _u16p), _p(wu, _u16p), _p(wd, _u16p),
        T, H, F, E, k, _p(tok, _i32p), 0 if tok is None else len(tok), _p(out, _u16p),
        _p(res["idx"], _i32p), _p(res["w"], _f32p), _p(res["cnt"], _i32p), _p(res["off"], _i32p),
        _p(res["perm"], _i32p), _p(res["pos"], _i32p), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle moe_layer rejected its arguments")
    res["out"] = out
    return res


def splitk_gemm(X, Wt, split, rows=None, nthreads=None):
    X, Wt = _u16(X), _u16(Wt)
    M, K = X.shape
    N = Wt.shape[0]
    r = _i32(rows)
    Y = np.empty((len(r) if r is not None else M, N), dtype=np.uint16)
    rc = lib().eto_splitk_gemm(_p(X, _u16p), _p(Wt, _u16p), M, N, K, split, _p(r, _i32p),
                               0 if r is None else len(r), _p(Y, _u16p),
                               nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle splitk_gemm rejected its arguments")
    return Y


def rmsnorm_row(x, gamma, eps):
    x, gamma = _u16(x), _u16(gamma)
    out = np.empty_like(x)
    lib().eto_rmsnorm_row(_p(x, _u16p), _p(gamma, _u16p), float(eps), x.shape[0], _p(out, _u16p))
    return out


def rmsnorm_row_f32(x, gamma, eps):
    """R15: the block's fp32 fixed-order RMSNorm of one row."""
    x, gamma = _u16(x), _u16(gamma)
    out = np.empty_like(x)
    lib().eto_rmsnorm_row_f32(_p(x, _u16p), _p(gamma, _u16p), float(eps), x.shape[0],
                              _p(out, _u16p))
    return out


def mlp_chain(x, gamma, eps, wg, wu, wd, rows=None, nthreads=None):
    x, gamma, wg, wu, wd = _u16(x), _u16(gamma), _u16(wg), _u16(wu), _u16(wd)
    B, H = x.shape
    F = wg.shape[0]
    r = _i32(rows)
    out = np.empty((len(r) if r is not None else B, H), dtype=np.uint16)
    rc = lib().eto_mlp_chain(_p(x, _u16p), _p(gamma, _u16p), float(eps), _p(wg, _u16p),
                             _p(wu, _u16p), _p(wd, _u16p), B, H, F, _p(r, _i32p),
                             0 if r is None else len(r), _p(out, _u16p),
                             nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle mlp_chain rejected its arguments")
    return out


def moe_block(x, gamma, eps, wr, bias, wg, wu, wd, sg=None, su=None, sd=None, k=2, tokens=None,
              nthreads=None):
    """The fused MoE block (R14): routing of x_hat = RMSNorm(x) * gamma, routed
    experts and the shared expert (sg/su [Fs,H], sd [H,Fs]; None = none) on x_hat,
    out = bf16(x + sum_j w_j y_j + y_s).  Returns dict(out, xhat, idx, w, cnt, perm)."""
    x, gamma, wr, wg, wu, wd = _u16(x), _u16(gamma), _u16(wr), _u16(wg), _u16(wu), _u16(wd)
    T, H = x.shape
    E, F, _ = wg.shape
    Fs = 0 if sg is None else _u16(sg).shape[0]
    sg, su, sd = (_u16(sg), _u16(su), _u16(sd)) if Fs else (None, None, None)
    tok = _i32(tokens)
    out = np.empty((len(tok) if tok is not None else T, H), dtype=np.uint16)
    res = dict(xhat=np.empty((T, H), np.uint16), idx=np.empty((T, k), np.int32),
               w=np.empty((T, k), np.float32), cnt=np.empty(E, np.int32),
               perm=np.empty(T * k, np.int32))
    b = _f32(bias)
    rc = lib().eto_moe_block(
        _p(x, _u16p), _p(gamma, _u16p), float(eps), _p(wr, _u16p), _p(b, _f32p), _p(wg, _u16p),
        _p(wu, _u16p), _p(wd, _u16p), _p(sg, _u16p), _p(su, _u16p), _p(sd, _u16p), T, H, F, Fs, E,
        k, _p(tok, _i32p), 0 if tok is None else len(tok), _p(out, _u16p), _p(res["xhat"], _u16p),
        _p(res["idx"], _i32p), _p(res["w"], _f32p), _p(res["cnt"], _i32p), _p(res["perm"], _i32p),
        nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle moe_block rejected its arguments")
    res["out"] = out
    return res
