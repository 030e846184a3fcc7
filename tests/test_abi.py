"""The C-ABI library without a GPU: it loads, exports every declared entry
point, sizes workspaces, and rejects invalid arguments before any device work."""
import ctypes
import os
import re

import pytest

from moe_task_scheduling_gb300 import etmoe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "etmoe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(et_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return etmoe.load()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "et_moe_layer" in names and "et_splitk_gemm" in names and "et_mlp_chain" in names
    raw = ctypes.CDLL(etmoe.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in etmoe.h but not exported"
    assert set(names) == set(etmoe.exported_symbols())


SOURCES = ("Prompt Boundary-Aware Scheduling with Event Tensors", "Megakernels ch. 5",
           "has no counterpart")


def declaration_blocks():
    """Each exported entry point's comment block: the last section comment
    ("/* ----") before its first declaration in etmoe.h, with everything up to
    the declaration (a block may cover several calls)."""
    text = open(HEADER).read()
    out = {}
    for name in declared_functions():
        m = re.search(r"\b" + name + r"\s*\(", text)
        before = text[:m.start()]
        block = before[before.rfind("/* ---"):]
        out[name] = " ".join(re.sub(r"^\s*\*", " ", block, flags=re.M).split())
    return out


def test_every_compute_entry_point_cites_its_source():
    """Each declaration of a compute call (and the calls the hot path consists
    of) carries, in its own comment block, the passage that defines it."""
    blocks = declaration_blocks()
    compute = [n for n in blocks if not n.endswith(("_workspace_bytes", "status", "_string",
                                                    "version"))]
    assert {"et_moe_layer", "et_splitk_gemm", "et_mlp_chain"} <= set(compute)
    for name in compute:
        assert any(src in blocks[name] for src in SOURCES), f"{name}: no source named"


def test_version_and_error_string(lib):
    assert lib.et_version() >= 100
    assert isinstance(lib.et_last_error_string(), bytes)


def test_workspace_sizes(lib):
    a = etmoe.et_moe_workspace_bytes(16, 256, 512, 8, 2)
    b = etmoe.et_moe_workspace_bytes(512, 4096, 14336, 8, 2)
    c = etmoe.et_moe_workspace_bytes(4096, 2048, 768, 128, 8)
    assert 0 < a < b and c > 0
    assert a % 256 == 0 and b % 256 == 0
    # the permuted activations, h and y buffers dominate: at least T*k*(2H+F)*2 bytes
    assert b >= 512 * 2 * (2 * 4096 + 14336) * 2
    assert etmoe.et_moe_workspace_bytes(16, 100, 512, 8, 2) == 0   # H not a multiple of 128
    assert etmoe.et_moe_workspace_bytes(16, 256, 512, 8, 9) == 0   # k > 8
    assert etmoe.et_moe_workspace_bytes(16, 256, 512, 2, 3) == 0   # k > E
    assert etmoe.et_moe_workspace_bytes(0, 256, 512, 8, 2) == 0
    assert etmoe.et_splitk_workspace_bytes(256, 4096, 14336, 8) >= 8 * 256 * 4096 * 4
    assert etmoe.et_splitk_workspace_bytes(256, 4096, 14336, 9) == 0  # K % (64*split) != 0
    assert etmoe.et_mlp_workspace_bytes(256, 4096, 14336) > 0
    assert etmoe.et_mlp_workspace_bytes(256, 4000, 14336) == 0


def _moe_call(lib, **over):
    args = dict(x=16, wr=16, bias=None, wg=16, wu=16, wd=16, out=16, idx=None, w=None, cnt=None,
                perm=None, T=4, dT=None, T_max=16, H=256, F=512, E=8, k=2, ws=256, wsb=1 << 30,
                opts=None, stream=None)
    args.update(over)
    return lib.et_moe_layer(*args.values())


def test_moe_validation(lib):
    E = etmoe
    assert _moe_call(lib, x=None) == E.ET_ERR_INVALID
    assert _moe_call(lib, H=100) == E.ET_ERR_UNSUPPORTED
    assert _moe_call(lib, k=9) == E.ET_ERR_UNSUPPORTED
    assert _moe_call(lib, E=300) == E.ET_ERR_UNSUPPORTED
    assert _moe_call(lib, T=17) == E.ET_ERR_INVALID
    assert _moe_call(lib, T=-1) == E.ET_ERR_INVALID
    assert _moe_call(lib, x=18) == E.ET_ERR_INVALID           # misaligned
    assert _moe_call(lib, ws=None) == E.ET_ERR_WORKSPACE
    assert _moe_call(lib, ws=512 + 8) == E.ET_ERR_WORKSPACE   # misaligned workspace
    assert _moe_call(lib, wsb=1024) == E.ET_ERR_WORKSPACE     # too small
    assert b"too small" in lib.et_last_error_string()
    # T == 0 with a host count: nothing to do, nothing launched
    assert _moe_call(lib, T=0) == E.ET_OK


def test_splitk_and_mlp_validation(lib):
    E = etmoe
    sk = lambda **o: lib.et_splitk_gemm(*dict(dict(X=16, W=16, Y=16, M=1, dM=None, Mm=8, N=256,  # noqa: E731
                                                    K=1024, s=8, ws=256, wsb=1 << 30, o=None,
                                                    st=None), **o).values())
    assert sk(K=1000) == E.ET_ERR_UNSUPPORTED
    assert sk(N=200) == E.ET_ERR_UNSUPPORTED
    assert sk(s=0) == E.ET_ERR_UNSUPPORTED
    assert sk(M=9) == E.ET_ERR_INVALID
    assert sk(Y=None) == E.ET_ERR_INVALID
    assert sk(wsb=16) == E.ET_ERR_WORKSPACE
    assert sk(M=0) == E.ET_OK
    mc = lambda **o: lib.et_mlp_chain(*dict(dict(x=16, g=16, eps=1e-5, wg=16, wu=16, wd=16,  # noqa: E731
                                                  out=16, B=2, dB=None, Bm=4, H=256, F=384,
                                                  ws=256, wsb=1 << 30, o=None, st=None),
                                             **o).values())
    assert mc(F=300) == E.ET_ERR_UNSUPPORTED
    assert mc(B=5) == E.ET_ERR_INVALID
    assert mc(eps=-1.0) == E.ET_ERR_INVALID
    assert mc(g=None) == E.ET_ERR_INVALID
    assert mc(B=0) == E.ET_OK


def test_status_rejects_null(lib):
    code = ctypes.c_int32()
    assert lib.et_status(None, None, ctypes.byref(code), None) == etmoe.ET_ERR_INVALID
    assert lib.et_reset_status(None, None) == etmoe.ET_ERR_INVALID
