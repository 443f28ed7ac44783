"""dflash_gemm_noalloc: the GEMM entry point that allocates no device memory.

It exists for callers that cannot call cudaMalloc (a loop that must not risk
the device synchronisation cudaMalloc/cudaFree can cause, a process whose
free memory a caching allocator holds, code next to a global-mode stream
capture). Its split-K scratch is a fixed array inside the library. Here it is
called through the C ABI twice in a row and compared with dflash_debug_gemm,
which allocates its own workspace. This file is collected last on purpose.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


@pytest.mark.parametrize("N,M,K,splits", [
    (4096, 16, 4096, 0),     # stream-K over the fixed partial buffer
    (1000, 40, 1024, 3),     # explicit split-K
    (20096, 100, 512, 0),    # 157 tiles of 128 tokens: the grid is cut to the 64 CTAs the buffer holds
    (4096, 256, 1024, 0),    # clusters of two CTA pairs exchanging half sums (no partials)
    (2048, 300, 512, 0),     # CTA pairs over 256-token tiles with a ragged token tail
])
def test_noalloc_gemm_matches_the_allocating_entry_point_twice(dfl, N, M, K, splits):
    """Two calls in a row (the second sees the first call's scratch contents),
    each equal to dflash_debug_gemm and to an fp32 matmul of the same bf16
    operands within the GEMM tests' tolerance."""
    lib = dfl.load_library()
    g = torch.Generator(device="cpu").manual_seed(N + M + K)
    Wh = torch.randn(N, K, generator=g).to(torch.bfloat16)
    Xh = torch.randn(M, K, generator=g).to(torch.bfloat16)
    exact = (Xh.float() @ Wh.float().T).to(DEV)
    W, X = Wh.to(DEV), Xh.to(DEV)
    ref = dfl.dflash_debug_gemm(W, X, splits=splits)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    tol = 1e-3 * np.sqrt(K)
    for _ in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        st = lib.dflash_gemm_noalloc(W.data_ptr(), X.data_ptr(), Y.data_ptr(), N, M, K, splits, stream)
        assert st == dfl.DFLASH_OK, lib.dflash_last_error(None)
        err = (Y - ref).abs().max().item()
        assert err <= tol, err
        err = (Y - exact).abs().max().item()
        assert err <= tol, err


def test_noalloc_gemm_rejects_scratch_overflow(dfl):
    lib = dfl.load_library()
    N, M, K = 8192, 256, 4096   # 16 splits x 256 x 8192 floats = 32 Mi floats > 2 Mi
    W = torch.zeros(N, K, dtype=torch.bfloat16, device=DEV)
    X = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    Y = torch.zeros(M, N, dtype=torch.float32, device=DEV)
    st = lib.dflash_gemm_noalloc(W.data_ptr(), X.data_ptr(), Y.data_ptr(), N, M, K, 16,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == dfl.DFLASH_EINVAL
    assert b"scratch" in lib.dflash_last_error(None)
