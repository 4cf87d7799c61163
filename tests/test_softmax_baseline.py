"""The exact-softmax comparator's conventions, on CPU tensors (math backend):
weights exp(q.k) with scale 1, the causal mask's orientation, the zero-padded
form, and the KV-cache decode step, each against the float64 oracle's exact
causal softmax. The GPU backends are checked against the same oracle in
tests/test_gpu_softmax_baseline.py."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from fixed_state_recurrence_phi_b300 import softmax_baseline as SB  # noqa: E402
from fixed_state_recurrence_phi_b300.inputs import np_qkv  # noqa: E402
from oracle import tsa_oracle as O  # noqa: E402


def _heads(B, H, N, d, dv, seed):
    qs, ks, vs = [], [], []
    for i in range(B * H):
        q, k, v = np_qkv(N, d, dv, (seed, i))
        qs.append(q); ks.append(k); vs.append(v)
    t = lambda xs: torch.tensor(np.stack(xs)).reshape(B, H, N, -1)
    return t(qs), t(ks), t(vs)


@pytest.mark.parametrize("padded", [False, True])
def test_prefill_is_the_oracle_softmax(padded):
    B, H, N, d, dv = 2, 2, 53, 16, 64
    q, k, v = _heads(B, H, N, d, dv, 11)
    c = SB.SoftmaxAttention(SB.SDPBackend.MATH, padded)
    out = c.prefill(c.keys(q, dv), c.keys(k, dv), v)
    assert out.shape == (B, H, N, dv)
    for b in range(B):
        for h in range(H):
            ref = O.softmax_attention(q[b, h].numpy(), k[b, h].numpy(), v[b, h].numpy())
            assert np.abs(out[b, h].numpy() - ref).max() < 1e-12


def test_prefill_is_causal_and_unscaled():
    N, d, dv = 20, 16, 32
    q, k, v = _heads(1, 1, N, d, dv, 12)
    c = SB.SoftmaxAttention(SB.SDPBackend.MATH)
    out = c.prefill(q, k, v)[0, 0]
    # row 0 attends to token 0 alone
    assert torch.allclose(out[0], v[0, 0, 0], atol=1e-15)
    # row 1: weights e^{q1.k0}, e^{q1.k1} (scale 1, not 1/sqrt(d))
    w = torch.exp(q[0, 0, 1] @ k[0, 0, :2].T)
    assert torch.allclose(out[1], (w @ v[0, 0, :2]) / w.sum(), atol=1e-14)
    # later tokens do not reach earlier rows
    v2 = v.clone()
    v2[..., 10:, :] += 100.0
    out2 = c.prefill(q, k, v2)[0, 0]
    assert torch.equal(out2[:10], out[:10]) and not torch.allclose(out2[10:], out[10:])


@pytest.mark.parametrize("padded", [False, True])
def test_decode_step_with_cache(padded):
    """Token pos's step writes its k, v into the cache and attends over
    tokens 0..pos: it equals row pos of the causal softmax over the prefix."""
    B, H, N, d, dv = 1, 3, 40, 16, 64
    q, k, v = _heads(B, H, N, d, dv, 13)
    c = SB.SoftmaxAttention(SB.SDPBackend.MATH, padded)
    kc, vc = c.cache(torch.zeros_like(k), torch.zeros_like(v))
    outs = [c.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], kc, vc, t) for t in range(N)]
    assert torch.equal(kc[..., :d], k) and torch.equal(vc, v)
    if padded:
        assert kc.shape[-1] == dv and not kc[..., d:].any()
    for h in range(H):
        ref = O.softmax_attention(q[0, h].numpy(), k[0, h].numpy(), v[0, h].numpy())
        got = torch.stack([o[0, h] for o in outs]).numpy()
        assert np.abs(got - ref).max() < 1e-12


def test_exponent_and_crossover_arithmetic():
    """The bench's fit and crossover on exact power laws: t_ours = a N and
    t_softmax = b N^2 cross at N = a / b, and log-log interpolation between
    sweep points is exact for power laws."""
    import bench
    ns = [256, 512, 1024, 2048, 4096, 8192]
    ours = [1e-3 * n for n in ns]
    soft = [1e-6 * n * n for n in ns]
    assert abs(bench.loglog_slope(ns, ours) - 1.0) < 1e-12
    assert abs(bench.loglog_slope(ns, soft) - 2.0) < 1e-12
    assert abs(bench.crossover_n(ns, ours, soft) - 1000.0) < 1e-6
    assert bench.crossover_n(ns, [1.0] * 6, [2.0] * 6) == 256          # faster everywhere
    assert bench.crossover_n(ns, [2.0] * 6, [1.0] * 6) is None         # never faster
    # a noisy win below the last crossing does not count
    assert abs(bench.crossover_n(ns, [1, 3, 3, 3, 1, 1], [2, 2, 2, 2, 2, 2]) - 2048 * 2 ** (
        np.log(2 / 3) / (np.log(2 / 3) - np.log(2)))) < 1e-6
