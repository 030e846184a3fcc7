"""The split-K entry point that allocates nothing, checked against the
workspace entry point on a GPU.

et_splitk_gemm_noalloc serves callers that cannot allocate device memory --
an op or plugin interface that hands the library only its inputs and
outputs, or a latency-critical path where cudaMalloc could synchronise the
device.  Its scratch is a fixed area inside the library that every call
reuses, so this checks two calls in a row (different shapes), each against
et_splitk_gemm with a caller workspace, and that a shape whose scratch does
not fit is refused before anything runs.  The file is named to be collected
last.
"""
import numpy as np
import pytest
import torch

from tests.helpers import assert_close_bf16
from moe_task_scheduling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    X = (torch.randn((M, K), generator=g, device="cuda")).to(torch.bfloat16)
    W = (torch.randn((N, K), generator=g, device="cuda") / np.sqrt(K)).to(torch.bfloat16)
    return X, W


def _with_workspace(etmoe, X, W, split):
    M, N, K = X.shape[0], W.shape[0], X.shape[1]
    ws = etmoe.alloc_workspace(etmoe.et_splitk_workspace_bytes(M, N, K, split))
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    etmoe.et_splitk_gemm(X, W, Y, split=split, workspace=ws)
    torch.cuda.synchronize()
    assert etmoe.et_status(ws)[0] == 0
    return Y


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_lib):
    # two calls in a row through the shared built-in scratch, different shapes
    for (M, N, K, split, seed) in ((64, 4096, 14336, 8, 71), (5, 256, 1024, 4, 72)):
        X, W = _inputs(M, N, K, seed)
        ref = _with_workspace(cuda_lib, X, W, split)
        Y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        cuda_lib.et_splitk_gemm_noalloc(X, W, Y, split=split)
        torch.cuda.synchronize()
        assert_close_bf16(wl.bits(Y), wl.bits(ref), f"no-alloc split-K M={M} N={N} K={K}")


def test_noalloc_refuses_shapes_beyond_its_scratch(cuda_lib):
    M, N, K, split = 256, 4096, 14336, 8  # needs ~32 MiB of partial sums
    assert cuda_lib.et_splitk_workspace_bytes(M, N, K, split) > (16 << 20)
    X, W = _inputs(M, N, K, 73)
    Y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    rc = cuda_lib.et_splitk_gemm_noalloc(X, W, Y, split=split, check=False)
    assert rc == cuda_lib.ET_ERR_WORKSPACE
    assert "scratch" in cuda_lib.last_error()
    torch.cuda.synchronize()
    assert torch.all(Y.float() == 7.0)
