"""The split-K entry point that allocates nothing, checked on a GPU.

et_splitk_gemm_noalloc serves callers that cannot allocate device memory --
an op or plugin interface that hands the library only its inputs and
outputs, or a latency-critical path where cudaMalloc could synchronise the
device.  Its scratch is a fixed area inside the library that every call
reuses, so this checks calls in a row of different shapes:
- each bit for bit against et_splitk_gemm with a caller workspace (the same
  kernel, tiles and split order, so the result must be identical);
- the device status of each call through et_splitk_noalloc_status;
- the largest shape whose scratch fits (M = 127 at N = 4096, K = 14336,
  split 8: the fp32 partials end 127 KB short of the area's end) and a small
  one, each also against the oracle;
- that a shape whose scratch does not fit is refused before anything runs.
The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from tests.helpers import assert_close_bf16
from moe_task_scheduling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SCRATCH = 16 << 20


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


# (M, N, K, split, seed, compare with the oracle): the largest shape that fits,
# a small one, then the first again -- so each call follows a different shape
CALLS = ((127, 4096, 14336, 8, 71, True), (5, 256, 1024, 4, 72, True),
         (64, 4096, 14336, 8, 73, False), (127, 4096, 14336, 8, 71, False))


def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row(cuda_lib, oracle):
    assert cuda_lib.et_splitk_workspace_bytes(127, 4096, 14336, 8) <= SCRATCH
    assert cuda_lib.et_splitk_workspace_bytes(128, 4096, 14336, 8) > SCRATCH
    for (M, N, K, split, seed, vs_oracle) in CALLS:
        X, W = _inputs(M, N, K, seed)
        ref = _with_workspace(cuda_lib, X, W, split)
        Y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        cuda_lib.et_splitk_gemm_noalloc(X, W, Y, split=split)
        assert cuda_lib.et_splitk_noalloc_status() == (0, 0)
        assert torch.equal(Y, ref), f"no-alloc split-K M={M} N={N} K={K} differs"
        if vs_oracle:
            want = oracle.splitk_gemm(wl.bits(X), wl.bits(W), split)
            assert_close_bf16(wl.bits(Y), want, f"no-alloc split-K M={M} N={N} K={K}")


def test_noalloc_refuses_shapes_beyond_its_scratch(cuda_lib):
    M, N, K, split = 256, 4096, 14336, 8  # needs ~32 MiB of partial sums
    assert cuda_lib.et_splitk_workspace_bytes(M, N, K, split) > SCRATCH
    X, W = _inputs(M, N, K, 74)
    Y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    rc = cuda_lib.et_splitk_gemm_noalloc(X, W, Y, split=split, check=False)
    assert rc == cuda_lib.ET_ERR_WORKSPACE
    assert "scratch" in cuda_lib.last_error()
    torch.cuda.synchronize()
    assert torch.all(Y.float() == 7.0)
