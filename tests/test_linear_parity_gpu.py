"""Parity of the tensor-core linear layer (ssm_linear_fwd; the block's
projections) against the exact fp64 product, across K from one partial
32-wide K block to the weight-gradient contraction over every row, with
ragged M and N tails, bias, residual and strided operands."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

# (M, N, K): ragged 128-row/column tiles, K below one block, K over many
# drain groups, and the block's own shapes.
SHAPES = [(1, 1, 1), (37, 5, 3), (200, 80, 48), (300, 257, 768), (16384 // 8, 1536, 1536),
          (130, 48, 16384), (2, 3, 4100)]


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("shape", SHAPES)
def test_linear_matches_fp64(lib, shape):
    import torch
    M, N, K = shape
    rng = np.random.Generator(np.random.PCG64(300 + SHAPES.index(shape)))
    X = rng.standard_normal((M, K), dtype=np.float32)
    W = (rng.standard_normal((N, K), dtype=np.float32) / np.float32(np.sqrt(K)))
    b = rng.standard_normal(N, dtype=np.float32)
    R = rng.standard_normal((M, N), dtype=np.float32)
    g = lambda a: torch.from_numpy(a).cuda()
    Y = lib.linear(g(X), g(W), g(b), g(R)).cpu().numpy().astype(np.float64)
    ref = X.astype(np.float64) @ W.astype(np.float64).T + b + R
    assert _rel(Y, ref) <= 2e-6, _rel(Y, ref)
    Y0 = lib.linear(g(X), g(W)).cpu().numpy().astype(np.float64)
    ref0 = X.astype(np.float64) @ W.astype(np.float64).T
    assert _rel(Y0, ref0) <= 2e-6, _rel(Y0, ref0)
    torch.cuda.synchronize()
    assert lib.ssm_device_faults() == 0


def test_linear_strided_and_in_place_residual(lib):
    import torch
    rng = np.random.Generator(np.random.PCG64(399))
    M, N, K = 260, 136, 200
    big = rng.standard_normal((M, K + 24), dtype=np.float32)
    W = rng.standard_normal((N, K), dtype=np.float32) / np.float32(np.sqrt(K))
    Yb = rng.standard_normal((M, N + 8), dtype=np.float32)
    tX = torch.from_numpy(big).cuda()[:, 8:8 + K]
    tY = torch.from_numpy(Yb).cuda()
    view = tY[:, 4:4 + N]
    before = Yb[:, 4:4 + N].astype(np.float64)
    ws = torch.empty(lib.ssm_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    lib.ssm_linear_fwd(tX, torch.from_numpy(W).cuda(), None, view, view, ws)
    got = tY.cpu().numpy().astype(np.float64)
    ref = big[:, 8:8 + K].astype(np.float64) @ W.astype(np.float64).T + before
    assert _rel(got[:, 4:4 + N], ref) <= 2e-6
    assert np.array_equal(got[:, :4], Yb[:, :4]) and np.array_equal(got[:, 4 + N:], Yb[:, 4 + N:])
