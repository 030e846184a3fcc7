"""Split-K GEMM through event counters vs the oracle (GPU)."""
import numpy as np
import pytest
import torch

from moe_task_scheduling_gb300 import workloads as wl
from tests.helpers import assert_close_bf16

pytestmark = pytest.mark.gpu


def _rand(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _run(etmoe, X, W, split, M=None, d_M=None, M_max=None, ws=None, Y=None):
    dev = torch.device("cuda")
    Mm = M_max or X.shape[0]
    if ws is None:
        ws = etmoe.alloc_workspace(etmoe.et_splitk_workspace_bytes(Mm, W.shape[0], W.shape[1], split))
    if Y is None:
        Y = torch.full((Mm, W.shape[0]), 7.0, dtype=torch.bfloat16, device=dev)
    etmoe.et_splitk_gemm(X, W, Y, split=split, M=M, d_M=d_M, M_max=Mm, workspace=ws)
    torch.cuda.synchronize()
    code, detail = etmoe.et_status(ws)
    assert code == 0, (code, detail)
    return Y, ws


@pytest.mark.parametrize("M,N,K,split", [
    (1, 128, 64, 1), (1, 256, 512, 8), (3, 128, 1024, 16), (17, 256, 1024, 4),
    (64, 384, 2048, 2), (129, 256, 1024, 8), (200, 128, 512, 1), (256, 256, 768, 3),
    (300, 256, 512, 2), (513, 128, 256, 4),
    # more tile tasks than CTAs (several per CTA), with the last arriver (M <= 32) or
    # reduce tasks over several row tiles
    (40, 16384, 1024, 4), (600, 4096, 2048, 8), (8, 32768, 256, 2), (100, 32768, 256, 2)])
def test_splitk_small_shapes(cuda_lib, oracle, M, N, K, split):
    X = _rand((M, K), 1.0, 1 + M)
    W = _rand((N, K), 1.0 / np.sqrt(K), 2 + N)
    Y, _ = _run(cuda_lib, X.cuda(), W.cuda(), split)
    ref = oracle.splitk_gemm(wl.bits(X), wl.bits(W), split)
    assert_close_bf16(wl.bits(Y), ref, f"Y M={M} N={N} K={K} split={split}")


def test_splitk_zero_input(cuda_lib):
    X = torch.zeros((5, 512), dtype=torch.bfloat16, device="cuda")
    W = _rand((256, 512), 1.0, 3).cuda()
    Y, _ = _run(cuda_lib, X, W, 8)
    assert torch.count_nonzero(Y.float()).item() == 0


def test_splitk_symbolic_M_one_workspace(cuda_lib, oracle):
    """One workspace, M read from device memory each call: M sweeps without any
    host-side change; rows >= M stay untouched; counters stay clean."""
    M_max, N, K, split = 96, 256, 1024, 8
    X = _rand((M_max, K), 1.0, 11)
    W = _rand((N, K), 1.0 / 32, 12)
    Xd, Wd = X.cuda(), W.cuda()
    ws = cuda_lib.alloc_workspace(cuda_lib.et_splitk_workspace_bytes(M_max, N, K, split))
    d_M = torch.zeros(1, dtype=torch.int32, device="cuda")
    for M in (1, 96, 33, 0, 64, 1):
        d_M.fill_(M)
        Y = torch.full((M_max, N), 7.0, dtype=torch.bfloat16, device="cuda")
        _run(cuda_lib, Xd, Wd, split, M=M_max, d_M=d_M, M_max=M_max, ws=ws, Y=Y)
        if M:
            ref = oracle.splitk_gemm(wl.bits(X[:M]), wl.bits(W), split)
            assert_close_bf16(wl.bits(Y[:M]), ref, f"Y M={M}")
        assert torch.all(Y[M:].float() == 7.0)
    assert torch.count_nonzero(ws[256:256 + 4 * 1 * (N // 128)]).item() == 0


def test_splitk_bounds_error_on_device_M(cuda_lib):
    M_max, N, K = 8, 128, 512
    ws = cuda_lib.alloc_workspace(cuda_lib.et_splitk_workspace_bytes(M_max, N, K, 2))
    d_M = torch.tensor([M_max + 1], dtype=torch.int32, device="cuda")
    X = torch.zeros((M_max, K), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((M_max, N), 7.0, dtype=torch.bfloat16, device="cuda")
    cuda_lib.et_splitk_gemm(X, W, Y, split=2, M=0, d_M=d_M, M_max=M_max, workspace=ws)
    code, _ = cuda_lib.et_status(ws)
    assert code == cuda_lib.ET_ERR_BOUNDS
    assert torch.all(Y.float() == 7.0)
    cuda_lib.et_reset_status(ws)
    assert cuda_lib.et_status(ws)[0] == 0


def test_splitk_full_size_sweep(cuda_lib, oracle):
    """The configured shape: Y[M,4096] = X[M,14336] W, split 8, M in {1,8,64,256}
    served by one compiled kernel and one workspace; every row vs the oracle."""
    cfg = wl.SPLITK
    inp = wl.splitk_inputs(cfg, device="cuda")
    Xh, Wh = wl.bits(inp["X"]), wl.bits(inp["Wt"])
    ws = cuda_lib.alloc_workspace(cuda_lib.et_splitk_workspace_bytes(cfg.M_max, cfg.N, cfg.K,
                                                                     cfg.split))
    d_M = torch.zeros(1, dtype=torch.int32, device="cuda")
    for M in cfg.M_sweep:
        d_M.fill_(M)
        Y, _ = _run(cuda_lib, inp["X"], inp["Wt"], cfg.split, M=cfg.M_max, d_M=d_M,
                    M_max=cfg.M_max, ws=ws)
        ref = oracle.splitk_gemm(Xh[:M], Wh, cfg.split)
        assert_close_bf16(wl.bits(Y)[:M], ref, f"Y M={M}")
        assert torch.all(Y[M:].float() == 7.0)


# ---------------------------------------------------------------- Cluster Launch Control variant

def _run_clc(etmoe, X, W, split, M=None, d_M=None, M_max=None, ws=None, Y=None):
    dev = torch.device("cuda")
    Mm = M_max or X.shape[0]
    if ws is None:
        ws = etmoe.alloc_workspace(etmoe.et_splitk_workspace_bytes(Mm, W.shape[0], W.shape[1], split))
    if Y is None:
        Y = torch.full((Mm, W.shape[0]), 7.0, dtype=torch.bfloat16, device=dev)
    etmoe.et_splitk_gemm_clc(X, W, Y, split=split, M=M, d_M=d_M, M_max=Mm, workspace=ws)
    torch.cuda.synchronize()
    code, detail = etmoe.et_status(ws)
    assert code == 0, (code, detail)
    return Y, ws


@pytest.mark.parametrize("M,N,K,split", [
    (1, 128, 64, 1), (1, 256, 512, 8), (3, 128, 1024, 16), (17, 256, 1024, 4),
    (129, 256, 1024, 8), (300, 256, 512, 2), (513, 128, 256, 4)])
def test_splitk_clc_small_shapes(cuda_lib, oracle, M, N, K, split):
    """The hardware work queue gives the oracle's result, and the same bits as
    the static schedule (same tiles, same split order)."""
    X = _rand((M, K), 1.0, 1 + M)
    W = _rand((N, K), 1.0 / np.sqrt(K), 2 + N)
    Xd, Wd = X.cuda(), W.cuda()
    Y, _ = _run_clc(cuda_lib, Xd, Wd, split)
    ref = oracle.splitk_gemm(wl.bits(X), wl.bits(W), split)
    assert_close_bf16(wl.bits(Y), ref, f"CLC Y M={M} N={N} K={K} split={split}")
    Ys, _ = _run(cuda_lib, Xd, Wd, split)
    assert torch.equal(Y, Ys), "CLC and static schedules differ"


def test_splitk_clc_symbolic_M_shared_workspace(cuda_lib, oracle):
    """M from device memory; the CLC and static calls alternate on one workspace,
    whose counters must stay clean for both."""
    M_max, N, K, split = 300, 256, 1024, 8
    X = _rand((M_max, K), 1.0, 21)
    W = _rand((N, K), 1.0 / 32, 22)
    Xd, Wd = X.cuda(), W.cuda()
    ws = cuda_lib.alloc_workspace(cuda_lib.et_splitk_workspace_bytes(M_max, N, K, split))
    d_M = torch.zeros(1, dtype=torch.int32, device="cuda")
    for M in (1, 300, 33, 0, 257, 64):
        d_M.fill_(M)
        Y = torch.full((M_max, N), 7.0, dtype=torch.bfloat16, device="cuda")
        _run_clc(cuda_lib, Xd, Wd, split, M=M_max, d_M=d_M, M_max=M_max, ws=ws, Y=Y)
        Ys = torch.full((M_max, N), 7.0, dtype=torch.bfloat16, device="cuda")
        _run(cuda_lib, Xd, Wd, split, M=M_max, d_M=d_M, M_max=M_max, ws=ws, Y=Ys)
        assert torch.equal(Y, Ys)
        if M:
            ref = oracle.splitk_gemm(wl.bits(X[:M]), wl.bits(W), split)
            assert_close_bf16(wl.bits(Y[:M]), ref, f"CLC Y M={M}")
        assert torch.all(Y[M:].float() == 7.0)
    hdr = ws[:256].view(torch.int32).cpu().numpy()
    assert np.all(hdr[2:] == 0)
    n_ev = -(-M_max // 256) * (N // 128)
    assert torch.count_nonzero(ws[256:256 + 4 * n_ev]).item() == 0


def test_splitk_clc_full_size(cuda_lib, oracle):
    """The configured shape through the hardware queue, every M of the sweep,
    every row vs the oracle."""
    cfg = wl.SPLITK
    inp = wl.splitk_inputs(cfg, device="cuda")
    Xh, Wh = wl.bits(inp["X"]), wl.bits(inp["Wt"])
    ws = cuda_lib.alloc_workspace(cuda_lib.et_splitk_workspace_bytes(cfg.M_max, cfg.N, cfg.K,
                                                                     cfg.split))
    d_M = torch.zeros(1, dtype=torch.int32, device="cuda")
    for M in cfg.M_sweep:
        d_M.fill_(M)
        Y, _ = _run_clc(cuda_lib, inp["X"], inp["Wt"], cfg.split, M=cfg.M_max, d_M=d_M,
                        M_max=cfg.M_max, ws=ws)
        ref = oracle.splitk_gemm(Xh[:M], Wh, cfg.split)
        assert_close_bf16(wl.bits(Y)[:M], ref, f"CLC Y M={M}")
        assert torch.all(Y[M:].float() == 7.0)
