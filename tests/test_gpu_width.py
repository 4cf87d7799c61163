"""The state's width on the GPU: the abstract's claim that the m-th state is
C(d+m-1, m) wide ("a bound confirmed by SVD"), checked with the features the
library itself builds (tsa_feature_map) for many unit keys:

  - the stacked full tensor powers k^{(x)m} (d^m columns) have numerical rank
    C(d+m-1, m): only the symmetric monomials are independent;
  - the library's order-m block phi_m(k) (exactly C(d+m-1, m) columns) has
    that rank too, and spans the same space: appending it to the full tensor
    powers does not raise the rank;
  - <phi_m(q), phi_m(k)> = (q.k)^m / m! on device (closed form), and the
    feature map equals the oracle's phi.
The ranks are computed on the device (torch.linalg.matrix_rank, float64)."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrence_phi_b300 import build
    build.build()
    import gpu_helpers
    return gpu_helpers


def _unit_rows(K, d, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn((K, d), generator=g, device="cuda", dtype=torch.float32)
    return x / torch.linalg.vector_norm(x, dim=1, keepdim=True)


@pytest.mark.parametrize("d,n", [(16, 4), (16, 5), (32, 3)])
def test_width_by_rank_of_stacked_features(G, d, n):
    T, O = G.T, G.O
    K = 2000
    x = _unit_rows(K, d, seed=11 + d)
    D = T.feature_dim(d, n)
    phi = torch.empty((K, D), device="cuda", dtype=torch.float32)
    T.feature_map(d, n, x, phi)
    torch.cuda.synchronize()
    # the oracle's feature map on a sample of the rows
    ref = O.phi(x[:64].double().cpu().numpy(), n)
    assert np.abs(phi[:64].double().cpu().numpy() - ref).max() <= 1e-6
    x64 = x.double()
    off = 0
    for m in range(n):
        w = math.comb(d + m - 1, m)
        block = phi[:, off:off + w].double()
        if m <= 3:   # the order-4 block (3,876 columns, 65,536 for the full power) is
            # checked through its exact enumeration (host test) and the closed form
            full = torch.ones((K, 1), device="cuda", dtype=torch.float64)
            for _ in range(m):   # the full tensor power, d^m columns
                full = torch.einsum("ka,kb->kab", full, x64).reshape(K, -1)
            r_full = int(torch.linalg.matrix_rank(full, rtol=1e-8).item())
            r_block = int(torch.linalg.matrix_rank(block, rtol=1e-5).item())
            r_both = int(torch.linalg.matrix_rank(torch.cat([full, block], dim=1), rtol=1e-5).item())
            assert r_full == w, (m, r_full, w)
            assert r_block == w, (m, r_block, w)
            assert r_both == w, (m, r_both, w)
        # <phi_m(q), phi_m(k)> = (q.k)^m / m! for pairs of the rows
        q_, k_ = block[: K // 2], block[K // 2:]
        dots = (x64[: K // 2] * x64[K // 2:]).sum(1)
        assert torch.allclose((q_ * k_).sum(1), dots ** m / math.factorial(m), rtol=1e-5, atol=1e-6), m
        off += w
    assert off == D
