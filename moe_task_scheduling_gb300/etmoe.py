"""Thin ctypes binding of libetmoe.so: the same entry points as include/etmoe.h.

Only argument marshalling happens here (tensors -> device pointers, the
current torch stream -> cudaStream_t).  Every step of the path runs in the
CUDA kernels of libetmoe.so.  If the library is missing, `load()` raises:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libetmoe.so")

ET_OK, ET_ERR_INVALID, ET_ERR_WORKSPACE, ET_ERR_UNSUPPORTED, ET_ERR_CUDA, ET_ERR_TIMEOUT, \
    ET_ERR_BOUNDS = range(7)

STATUS_NAMES = {0: "ET_OK", 1: "ET_ERR_INVALID", 2: "ET_ERR_WORKSPACE", 3: "ET_ERR_UNSUPPORTED",
                4: "ET_ERR_CUDA", 5: "ET_ERR_TIMEOUT", 6: "ET_ERR_BOUNDS"}


class et_opts(ctypes.Structure):
    _fields_ = [("timeout_us", ctypes.c_uint32), ("trace_cap", ctypes.c_uint32),
                ("fault_mode", ctypes.c_int32), ("fault_arg", ctypes.c_int32),
                ("trace", ctypes.c_void_p)]


class et_moe_layer_desc(ctypes.Structure):
    _fields_ = [("gamma", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("w_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("ws_gate", ctypes.c_void_p), ("ws_up", ctypes.c_void_p),
                ("ws_down", ctypes.c_void_p), ("Fs", ctypes.c_int32), ("out", ctypes.c_void_p),
                ("x_hat", ctypes.c_void_p), ("topk_idx", ctypes.c_void_p),
                ("topk_w", ctypes.c_void_p), ("expert_counts", ctypes.c_void_p),
                ("perm", ctypes.c_void_p)]


class EtError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None
_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t

_SIGNATURES = {
    "et_version": (_i, []),
    "et_last_error_string": (ctypes.c_char_p, []),
    "et_moe_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "et_moe_layer": (_i, [_vp] * 11 + [_i, _vp] + [_i] * 5 + [_vp, _sz, _vp, _vp]),
    "et_moe_block_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "et_moe_block": (_i, [_vp, _vp, ctypes.c_float] + [_vp] * 8 + [_i] + [_vp] * 6 + [_i, _vp] +
                     [_i] * 5 + [_vp, _sz, _vp, _vp]),
    "et_moe_chain_workspace_bytes": (_sz, [_i, _vp, _i, _i, _i, _i, _i]),
    "et_moe_chain": (_i, [_i, _vp, _vp, _i, _vp] + [_i] * 5 + [_vp, _sz, _vp, _vp]),
    "et_splitk_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "et_splitk_gemm": (_i, [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _vp, _sz, _vp, _vp]),
    "et_splitk_gemm_noalloc": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "et_splitk_gemm_clc": (_i, [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _vp, _sz, _vp, _vp]),
    "et_mlp_workspace_bytes": (_sz, [_i, _i, _i]),
    "et_mlp_chain": (_i, [_vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _vp,
                          _sz, _vp, _vp]),
    "et_splitk_noalloc_status": (_i, [_vp, ctypes.POINTER(ctypes.c_int32),
                                      ctypes.POINTER(ctypes.c_int32)]),
    "et_status": (_i, [_vp, _vp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "et_reset_status": (_i, [_vp, _vp]),
}


def load(path: Optional[str] = None):
    """Open libetmoe.so (building nothing); raises if it is not there."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libetmoe.so not found at {p}: run __graft_entry__.build() first "
                           "(there is no CPU fallback for the CUDA path)")
    L = ctypes.CDLL(p)
    for name, (res, args) in _SIGNATURES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def exported_symbols():
    return list(_SIGNATURES)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _opts(timeout_us=0, fault_mode=0, fault_arg=0, trace=None):
    if not (timeout_us or fault_mode or trace is not None):
        return None
    cap = 0 if trace is None else (trace.numel() * trace.element_size() - 32) // 32
    return ctypes.byref(et_opts(timeout_us, cap, fault_mode, fault_arg, _ptr(trace)))


def alloc_trace(records: int, device="cuda"):
    """A zeroed device buffer for `records` trace records (see et_opts.trace)."""
    import torch
    return torch.zeros(32 + 32 * records, dtype=torch.uint8, device=device)


def read_trace(buf):
    """Decode a trace buffer: list of (type, role, a, b, cta, t_begin_ns, t_end_ns).
    The records sit in per-CTA shares of the buffer; unused slots are zero."""
    import numpy as np
    raw = buf.cpu().numpy()
    cap = (raw.size - 32) // 32
    rec = raw[32:32 + 32 * cap].reshape(-1, 32)
    ints = rec[:, :16].copy().view(np.int32).reshape(-1, 4)
    ts = rec[:, 16:].copy().view(np.uint64).reshape(-1, 2)
    return [(int(i[0]) & 0xff, int(i[0]) >> 8, int(i[1]), int(i[2]), int(i[3]), int(t[0]), int(t[1]))
            for i, t in zip(ints, ts) if t[1] != 0]


def _check(rc):
    if rc != ET_OK:
        raise EtError(rc, load().et_last_error_string().decode())


def last_error() -> str:
    return load().et_last_error_string().decode()


# ------------------------------------------------------------------ workspaces

def et_moe_workspace_bytes(T_max, H, F, E, k) -> int:
    return load().et_moe_workspace_bytes(T_max, H, F, E, k)


def et_moe_block_workspace_bytes(T_max, H, F, E, k, Fs) -> int:
    return load().et_moe_block_workspace_bytes(T_max, H, F, E, k, Fs)


def et_splitk_workspace_bytes(M_max, N, K, split) -> int:
    return load().et_splitk_workspace_bytes(M_max, N, K, split)


def et_mlp_workspace_bytes(B_max, H, F) -> int:
    return load().et_mlp_workspace_bytes(B_max, H, F)


def alloc_workspace(nbytes: int, device="cuda"):
    """A zeroed, 256-byte aligned byte buffer (torch owns the memory)."""
    import torch
    if nbytes <= 0:
        raise ValueError("invalid workspace size (shape rejected by the library)")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ compute calls

def et_moe_layer(x, w_router, router_bias, w_gate, w_up, w_down, out, *, k, T=None, d_T=None,
                 T_max=None, topk_idx=None, topk_w=None, expert_counts=None, perm=None,
                 workspace, stream=None, timeout_us=0, fault_mode=0, fault_arg=0, trace=None,
                 check=True):
    H = x.shape[1]
    E = w_router.shape[1]
    F = w_gate.shape[1]
    T_max = T_max if T_max is not None else x.shape[0]
    T = T if T is not None else x.shape[0]
    rc = load().et_moe_layer(
        _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
        _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(expert_counts), _ptr(perm), T, _ptr(d_T),
        T_max, H, F, E, k, _ptr(workspace), workspace.numel() if hasattr(workspace, "numel") else 0,
        _opts(timeout_us, fault_mode, fault_arg, trace), _stream(stream))
    if check:
        _check(rc)
    return rc


def et_moe_block(x, gamma, eps, w_router, router_bias, w_gate, w_up, w_down, ws_gate, ws_up,
                 ws_down, out, *, k, x_hat=None, T=None, d_T=None, T_max=None, topk_idx=None,
                 topk_w=None, expert_counts=None, perm=None, workspace, stream=None, timeout_us=0,
                 fault_mode=0, fault_arg=0, trace=None, check=True):
    H = x.shape[1]
    E = w_router.shape[1]
    F = w_gate.shape[1]
    Fs = 0 if ws_gate is None else ws_gate.shape[0]
    T_max = T_max if T_max is not None else x.shape[0]
    T = T if T is not None else x.shape[0]
    rc = load().et_moe_block(
        _ptr(x), _ptr(gamma), float(eps), _ptr(w_router), _ptr(router_bias), _ptr(w_gate),
        _ptr(w_up), _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down), Fs, _ptr(out),
        _ptr(x_hat), _ptr(topk_idx), _ptr(topk_w), _ptr(expert_counts), _ptr(perm), T, _ptr(d_T),
        T_max, H, F, E, k, _ptr(workspace), workspace.numel() if hasattr(workspace, "numel") else 0,
        _opts(timeout_us, fault_mode, fault_arg, trace), _stream(stream))
    if check:
        _check(rc)
    return rc


def layer_desc(w_router, router_bias, w_gate, w_up, w_down, out, *, gamma=None, eps=1e-5,
               ws_gate=None, ws_up=None, ws_down=None, x_hat=None, topk_idx=None, topk_w=None,
               expert_counts=None, perm=None):
    """One layer of et_moe_chain (gamma given: a fused block)."""
    return et_moe_layer_desc(
        _ptr(gamma), float(eps), _ptr(w_router), _ptr(router_bias), _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down),
        0 if ws_gate is None else ws_gate.shape[0], _ptr(out), _ptr(x_hat), _ptr(topk_idx),
        _ptr(topk_w), _ptr(expert_counts), _ptr(perm))


def _desc_array(layers):
    arr = (et_moe_layer_desc * len(layers))(*layers)
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def et_moe_chain_workspace_bytes(layers, T_max, H, F, E, k) -> int:
    arr, ptr = _desc_array(layers)
    return load().et_moe_chain_workspace_bytes(len(layers), ptr, T_max, H, F, E, k)


def et_moe_chain(layers, x, *, H, F, E, k, T=None, d_T=None, T_max=None, workspace, stream=None,
                 timeout_us=0, fault_mode=0, fault_arg=0, trace=None, check=True):
    """Chained layers in one launch: layers[l + 1] reads layers[l].out."""
    T_max = T_max if T_max is not None else x.shape[0]
    T = T if T is not None else x.shape[0]
    arr, ptr = _desc_array(layers)
    rc = load().et_moe_chain(len(layers), ptr, _ptr(x), T, _ptr(d_T), T_max, H, F, E, k,
                             _ptr(workspace),
                             workspace.numel() if hasattr(workspace, "numel") else 0,
                             _opts(timeout_us, fault_mode, fault_arg, trace), _stream(stream))
    if check:
        _check(rc)
    return rc


def et_splitk_gemm(X, Wt, Y, *, split, M=None, d_M=None, M_max=None, workspace, stream=None,
                   timeout_us=0, trace=None, check=True):
    K = X.shape[1]
    N = Wt.shape[0]
    M_max = M_max if M_max is not None else X.shape[0]
    M = M if M is not None else X.shape[0]
    rc = load().et_splitk_gemm(_ptr(X), _ptr(Wt), _ptr(Y), M, _ptr(d_M), M_max, N, K, split,
                               _ptr(workspace), workspace.numel(), _opts(timeout_us, trace=trace),
                               _stream(stream))
    if check:
        _check(rc)
    return rc


def et_splitk_gemm_clc(X, Wt, Y, *, split, M=None, d_M=None, M_max=None, workspace, stream=None,
                       timeout_us=0, check=True):
    """Split-K GEMM with the Cluster Launch Control work queue (same results)."""
    K = X.shape[1]
    N = Wt.shape[0]
    M_max = M_max if M_max is not None else X.shape[0]
    M = M if M is not None else X.shape[0]
    rc = load().et_splitk_gemm_clc(_ptr(X), _ptr(Wt), _ptr(Y), M, _ptr(d_M), M_max, N, K, split,
                                   _ptr(workspace), workspace.numel(), _opts(timeout_us),
                                   _stream(stream))
    if check:
        _check(rc)
    return rc


def et_splitk_gemm_noalloc(X, Wt, Y, *, split, M=None, stream=None, check=True):
    """Split-K GEMM with the library's built-in scratch (no workspace, no allocation)."""
    K = X.shape[1]
    N = Wt.shape[0]
    M = M if M is not None else X.shape[0]
    rc = load().et_splitk_gemm_noalloc(_ptr(X), _ptr(Wt), _ptr(Y), M, N, K, split, _stream(stream))
    if check:
        _check(rc)
    return rc


def et_splitk_noalloc_status(stream=None):
    """(code, detail) of the last no-alloc split-K call on this device (synchronises)."""
    code = ctypes.c_int32(0)
    detail = ctypes.c_int32(0)
    _check(load().et_splitk_noalloc_status(_stream(stream), ctypes.byref(code),
                                           ctypes.byref(detail)))
    return code.value, detail.value


def et_mlp_chain(x, gamma, eps, w_gate, w_up, w_down, out, *, B=None, d_B=None, B_max=None,
                 workspace, stream=None, timeout_us=0, fault_mode=0, fault_arg=0, trace=None,
                 check=True):
    H = x.shape[1]
    F = w_gate.shape[0]
    B_max = B_max if B_max is not None else x.shape[0]
    B = B if B is not None else x.shape[0]
    rc = load().et_mlp_chain(_ptr(x), _ptr(gamma), float(eps), _ptr(w_gate), _ptr(w_up),
                             _ptr(w_down), _ptr(out), B, _ptr(d_B), B_max, H, F, _ptr(workspace),
                             workspace.numel(), _opts(timeout_us, fault_mode, fault_arg, trace),
                             _stream(stream))
    if check:
        _check(rc)
    return rc


def et_status(workspace, stream=None):
    """(code, detail) of the workspace's sticky device status (synchronises)."""
    code = ctypes.c_int32(0)
    detail = ctypes.c_int32(0)
    _check(load().et_status(_ptr(workspace), _stream(stream), ctypes.byref(code),
                            ctypes.byref(detail)))
    return code.value, detail.value


def et_reset_status(workspace, stream=None):
    _check(load().et_reset_status(_ptr(workspace), _stream(stream)))
