"""The tcgen05 row-gathered GEMM against a float64 matmul of the same bf16
operands (needs a GB300): live row counts around the 16-row MMA step, the
64-row TMA box and the 256-row tile, K splits, and the count read on the
device."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sf():
    from sparse_reuse_gb300 import build
    build.build()
    import sparse_reuse_gb300 as m
    return m


def _run(sf, M, K, rows_cap, count, splits, on_device=True, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    X = (torch.randn((rows_cap, K), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    W = (torch.randn((M, K), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    Y = torch.full((rows_cap, M), float("nan"), device="cuda")
    cnt = torch.tensor([count], dtype=torch.int32, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    sf.sfk_gemm_bf16(None, X.data_ptr(), rows_cap, W.data_ptr(), M, K, cnt.data_ptr() if on_device else None,
                     count, Y.data_ptr(), M, splits, err.data_ptr())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = X[:count].double().cpu().numpy() @ W.double().cpu().numpy().T
    got = Y[:count].double().cpu().numpy()
    scale = np.abs(X[:count].double().cpu().numpy()) @ np.abs(W.double().cpu().numpy().T) + 1e-30
    assert np.all(np.abs(got - ref) <= 1e-4 * scale + 1e-6), np.max(np.abs(got - ref) / scale)
    assert torch.isnan(Y[count:]).all()                # rows past the count are untouched
    return Y


@pytest.mark.parametrize("count", [1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 288, 511])
def test_counts_single_split(sf, count):
    _run(sf, 256, 512, 512, count, 1)


@pytest.mark.parametrize("splits", [2, 3, 4, 5, 6, 7, 8])
def test_split_k(sf, splits):
    _run(sf, 384, 1536, 300, 288, splits)
    _run(sf, 384, 1536, 300, 50, splits, seed=1)
    _run(sf, 128, 1024, 256, 256, splits, seed=2)


def test_zero_rows_writes_nothing(sf):
    _run(sf, 128, 128, 64, 0, 1)
    _run(sf, 128, 128, 64, 0, 2)


def test_dense_count_and_long_k(sf):
    _run(sf, 128, 8960, 64, 50, 8, on_device=False)
    _run(sf, 1536, 1536, 288, 288, 4, on_device=False)


@pytest.mark.parametrize("count", [257, 300, 513])
@pytest.mark.parametrize("splits", [1, 3])
def test_dense_counts_split_into_equal_tiles(sf, count, splits):
    # a host-known count is cut into ceil(count / 256) tiles of equal size (a
    # multiple of 16); the last tile's row boxes reach past rows_cap (zero fill)
    _run(sf, 256, 512, count, count, splits, on_device=False, seed=4)


def test_split_results_are_deterministic(sf):
    a = _run(sf, 256, 2048, 288, 288, 6, seed=3)
    b = _run(sf, 256, 2048, 288, 288, 6, seed=3)
    assert torch.equal(a[:288], b[:288])


def test_bad_arguments_rejected(sf):
    # every buffer is real and larger than any launch these arguments describe
    X = torch.zeros((256, 1024), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((256, 1024), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((256, 256), device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    x, w, y, e = X.data_ptr(), W.data_ptr(), Y.data_ptr(), err.data_ptr()
    with pytest.raises(sf.SpecFoldError):
        sf.sfk_gemm_bf16(None, x, 64, w, 100, 64, None, 1, y, 100, 1, e)       # M not a multiple of 128
    with pytest.raises(sf.SpecFoldError):
        sf.sfk_gemm_bf16(None, x, 64, w, 128, 64, None, 1, y, 128, 2, e)       # more splits than K blocks
    with pytest.raises(sf.SpecFoldError):
        sf.sfk_gemm_bf16(None, x, 64, w, 128, 1024, None, 1, y, 128, 9, e)     # cluster larger than 8
    with pytest.raises(sf.SpecFoldError):
        sf.sfk_gemm_bf16(None, x, 64, w, 128, 1024, None, 1, y, 128, 0, e)     # no split at all
    torch.cuda.synchronize()
    assert int(err.item()) == 0