"""The exact-softmax comparator on the GPU (the library's fast attention
backends) against the float64 oracle's exact causal softmax, and the
truncated-Taylor prefill against it: the difference between the two GPU
results must be the oracle's own truncation error, element by element within
the parity tolerance."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrence_phi_b300 import build
    build.build()
    import gpu_helpers
    return gpu_helpers


def _sb():
    from fixed_state_recurrence_phi_b300 import softmax_baseline as SB
    return SB


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_every_backend_that_runs_is_the_oracle_softmax(G, dtype):
    SB = _sb()
    cfg = G.T.Config(1, 2, 16, 64, 3, dtype)
    N = 300
    q, k, v = G.make_inputs(cfg, N, seed=901)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    refs = [G.O.softmax_attention(qh[0, h], kh[0, h], vh[0, h]) for h in range(2)]
    ran = 0
    for c in SB.candidates(q.device):
        try:
            out = c.prefill(c.keys(q, 64), c.keys(k, 64), v)
        except RuntimeError:
            continue                       # this backend does not take these inputs
        ran += 1
        og = G.host(out)
        for h in range(2):
            e = G.rel_err(og[0, h], refs[h])
            assert e <= G.TOL[dtype], f"{c.name} head {h}: {e:.3e}"
    assert ran >= 1
    best, tried = SB.select(q, k, v)
    assert best.name in tried and isinstance(tried[best.name], float)


def test_decode_step_is_the_last_row(G):
    SB = _sb()
    cfg = G.T.Config(2, 4, 16, 64, 3, "bf16")
    N = 513
    q, k, v = G.make_inputs(cfg, N, seed=902)
    c, _ = SB.select(q[:, :, -1:], k, v, causal=False)
    kc, vc = c.cache(torch.zeros_like(k), torch.zeros_like(v))
    kc[:, :, : N - 1, :16] = k[:, :, : N - 1]
    vc[:, :, : N - 1] = v[:, :, : N - 1]
    o = G.host(c.decode_step(q[:, :, -1], k[:, :, -1], v[:, :, -1], kc, vc, N - 1))
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for b, h in G.sample_heads(2, 4, k=3, seed=5):
        # one query against all N keys: the oracle's last causal row
        full = G.O.softmax_attention(qh[b, h], kh[b, h], vh[b, h])[-1]
        assert G.rel_err(o[b, h], full) <= G.TOL["bf16"], (b, h)


def test_taylor_minus_softmax_is_the_truncation_error(G):
    """(tsa prefill - GPU softmax) equals (oracle Taylor - oracle softmax):
    the GPU paths differ by exactly the method's truncation, nothing else."""
    SB = _sb()
    cfg = G.T.Config(1, 2, 16, 64, 2, "f32")   # n = 2: a truncation error well above fp32 rounding
    N = 700
    q, k, v = G.make_inputs(cfg, N, seed=903)
    out, _ = G.gpu_prefill(cfg, q, k, v)
    c, _ = SB.select(q, k, v)
    sm = c.prefill(c.keys(q, 64), c.keys(k, 64), v)
    d_gpu = G.host(out) - G.host(sm)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for h in range(2):
        o_t, _ = G.oracle_prefill(qh[0, h], kh[0, h], vh[0, h], 2)
        d_ref = o_t - G.O.softmax_attention(qh[0, h], kh[0, h], vh[0, h])
        scale = np.abs(o_t).max()
        assert np.abs(d_ref).max() > 1e-3 * scale          # the truncation is visible
        assert np.abs(d_gpu[0, h] - d_ref).max() <= G.TOL["f32"] * scale, h
