"""Parity of the tensor-core prefill path (bf16 q, k, v; tcgen05 MMAs with fp32
TMEM accumulators) with the float64 oracle on the same seeded inputs: ragged
tails around the 128-token chunk, several spans per head (span-state pass and
scan), several value-column slices, continuation with ACCUMULATE, and
determinism. Tolerance: normwise relative error per head <= 2e-2 (bf16 inputs,
fp32 accumulation and states)."""
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


def _check_all_heads(G, cfg, N, seed, chunked=None):
    O = G.O
    q, k, v = G.make_inputs(cfg, N, seed)
    out, st = G.gpu_prefill(cfg, q, k, v)
    G.T.sync_status()
    Sg = G.canonical(cfg, st)
    og = G.host(out)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    worst = 0.0
    for b in range(cfg.B):
        for h in range(cfg.H):
            o_r, S_r = G.oracle_prefill(qh[b, h], kh[b, h], vh[b, h], cfg.n_terms, chunked=chunked)
            e = G.check_head(cfg, og[b, h], Sg[b, h], o_r, S_r, G.TOL["bf16"], f"N={N} b={b} h={h}")
            worst = max(worst, max(e))
    return worst


def test_bf16_uses_tensor_core_path(G):
    T = G.T
    for d, dv, n in [(16, 64, 3), (16, 64, 4), (32, 128, 3), (16, 128, 3), (32, 64, 2), (16, 32, 1)]:
        p = T.prefill_plan(T.Config(2, 4, d, dv, n, "bf16"), 4096)
        assert p["path"] == T.TSA_PATH_TC and p["chunk"] == 128, (d, dv, n, p)
    # fp32 inputs: split-bf16 tensor-core path where one CTA holds the head,
    # the CUDA-core path otherwise
    assert T.prefill_plan(T.Config(1, 8, 16, 64, 3, "f32"), 8192)["path"] == T.TSA_PATH_TC_F32
    assert T.prefill_plan(T.Config(1, 1, 16, 64, 3, "f32"), 256)["path"] == T.TSA_PATH_TC_F32
    assert T.prefill_plan(T.Config(1, 2, 16, 64, 4, "f32"), 333)["path"] == T.TSA_PATH_SIMT


@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 256, 257, 1000])
def test_tc_ragged_lengths(G, N):
    cfg = G.T.Config(2, 3, 16, 64, 3, "bf16", chunk=128)
    _check_all_heads(G, cfg, N, seed=200 + N)


@pytest.mark.parametrize("d,dv,n,N", [
    (16, 64, 4, 700),     # 8 feature blocks: a CTA pair, 4 blocks each
    (32, 128, 3, 600),    # 5 feature blocks: a CTA pair, the last block split by columns
    (32, 64, 3, 450),     # the same split at d_v 64
    (16, 128, 3, 500),    # one slice of 128 (+ the normaliser group: N = 144)
    (32, 32, 2, 400),     # one feature block
    (16, 32, 1, 300),     # n = 1: a running mean
])
def test_tc_slicing_shapes(G, d, dv, n, N):
    cfg = G.T.Config(1, 2, d, dv, n, "bf16")
    _check_all_heads(G, cfg, N, seed=300 + d + dv + n)


def test_tc_multi_span(G):
    """Few heads and a long sequence: the plan cuts each head into spans, so
    the span-state pass, the scan and the prefix-state readout all run."""
    cfg = G.T.Config(1, 2, 16, 64, 3, "bf16")
    plan = G.T.prefill_plan(cfg, 8192)
    assert plan["n_spans"] > 1 and plan["launches"] == 3
    _check_all_heads(G, cfg, 8192, seed=31, chunked=256)


def test_tc_multi_span_multi_slice_order4(G):
    """Order 4 with few heads: the value-sliced span pass and the scan, then
    the CTA-pair output pass starting each span from its prefix."""
    cfg = G.T.Config(1, 1, 16, 64, 4, "bf16")
    plan = G.T.prefill_plan(cfg, 5000)
    assert plan["n_spans"] > 1 and plan["cluster"] == 2
    _check_all_heads(G, cfg, 5000, seed=32, chunked=256)


def test_pair_plans(G):
    """The heads whose state one SM's tensor memory holds only in value slices
    are shared by a CTA pair: order 4 at d_k 16 (8 feature blocks, 4 each),
    d_k 32 (5 blocks: 2 each and the last split by columns)."""
    T = G.T
    for d, dv, n in [(16, 64, 4), (32, 128, 3), (32, 64, 3)]:
        p = T.prefill_plan(T.Config(4, 16, d, dv, n, "bf16"), 32768)
        assert p["path"] == T.TSA_PATH_TC and p["cluster"] == 2 and p["n_slices"] == 1, (d, dv, n, p)
    for d, dv, n in [(16, 64, 3), (16, 128, 3), (32, 32, 3)]:
        assert T.prefill_plan(T.Config(4, 16, d, dv, n, "bf16"), 32768)["cluster"] == 1


@pytest.mark.parametrize("d,dv,n,N", [
    (16, 64, 4, 1), (16, 64, 4, 127), (16, 64, 4, 129), (16, 64, 4, 385),
    (32, 128, 3, 1), (32, 128, 3, 200), (32, 64, 3, 500), (32, 64, 3, 129),
])
def test_pair_ragged(G, d, dv, n, N):
    cfg = G.T.Config(1, 3, d, dv, n, "bf16")
    _check_all_heads(G, cfg, N, seed=400 + d + dv + n + N)


@pytest.mark.parametrize("d,dv,n", [(16, 64, 4), (32, 128, 3)])
def test_pair_accumulate_continues_the_sequence(G, d, dv, n):
    T, O = G.T, G.O
    cfg = T.Config(1, 2, d, dv, n, "bf16")
    q, k, v = G.make_inputs(cfg, 900, seed=35 + d)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    _, st = G.gpu_prefill(cfg, sl(q, 0, 333), sl(k, 0, 333), sl(v, 0, 333))
    out2, st = G.gpu_prefill(cfg, sl(q, 333, 900), sl(k, 333, 900), sl(v, 333, 900), states=st,
                             accumulate=True)
    Sg = G.canonical(cfg, st)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for h in range(2):
        o_r, S_r = O.prefill_recurrent(qh[0, h], kh[0, h], vh[0, h], n)
        G.check_head(cfg, G.host(out2)[0, h], Sg[0, h], o_r[333:], S_r, G.TOL["bf16"], "accumulate")


def test_tc_accumulate_continues_the_sequence(G):
    T, O = G.T, G.O
    cfg = T.Config(1, 2, 16, 64, 3, "bf16")
    q, k, v = G.make_inputs(cfg, 1500, seed=33)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    _, st = G.gpu_prefill(cfg, sl(q, 0, 650), sl(k, 0, 650), sl(v, 0, 650))
    out2, st = G.gpu_prefill(cfg, sl(q, 650, 1500), sl(k, 650, 1500), sl(v, 650, 1500), states=st,
                             accumulate=True)
    Sg = G.canonical(cfg, st)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for h in range(2):
        o_r, S_r = O.prefill_recurrent(qh[0, h], kh[0, h], vh[0, h], 3)
        G.check_head(cfg, G.host(out2)[0, h], Sg[0, h], o_r[650:], S_r, G.TOL["bf16"], "accumulate")


def test_tc_deterministic_and_padding_zero(G):
    T = G.T
    cfg = T.Config(1, 4, 16, 64, 4, "bf16")
    q, k, v = G.make_inputs(cfg, 3000, seed=34)
    o1, s1 = G.gpu_prefill(cfg, q, k, v)
    o2, s2 = G.gpu_prefill(cfg, q, k, v)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    D, Dp = T.feature_dim(16, 4), T.state_pad_dim(16, 4)
    st = s1.view(4, Dp * 65)
    S = st[:, :Dp * 64].view(4, Dp, 64)
    z = st[:, Dp * 64:]
    assert torch.count_nonzero(S[:, D:]) == 0 and torch.count_nonzero(z[:, D:]) == 0
    T.sync_status()


def test_append_plans(G):
    """Segments of 17 to 64 tokens of a state of at most two feature blocks
    (d_v <= 64) take the single-chunk append form: three CTAs per SM, at most
    ~75 KB of shared memory each."""
    T = G.T
    for d, dv, n in [(16, 64, 3), (32, 64, 2), (16, 32, 1)]:
        for N in (17, 33, 64):
            p = T.prefill_plan(T.Config(64, 16, d, dv, n, "bf16"), N, num_sms=148)
            assert p["path"] == T.TSA_PATH_TC and p["ctas_per_sm"] == 3, (d, dv, n, N, p)
            assert p["smem_bytes"] + 1024 <= 228 * 1024 // 3 and p["n_spans"] == 1
        assert T.prefill_plan(T.Config(64, 16, d, dv, n, "bf16"), 65, num_sms=148)["ctas_per_sm"] == 1
    # a state one CTA holds only in value slices (or with a pair) keeps the full form
    assert T.prefill_plan(T.Config(1, 2, 32, 64, 3, "bf16"), 64, num_sms=148)["cluster"] == 2
    assert T.prefill_plan(T.Config(1, 2, 16, 128, 3, "bf16"), 64, num_sms=148)["ctas_per_sm"] == 1


@pytest.mark.parametrize("d,dv,n,N", [(16, 64, 3, 17), (16, 64, 3, 64), (16, 32, 3, 40), (16, 32, 2, 33),
                                      (32, 64, 2, 50), (32, 32, 1, 21)])
def test_append_form_from_zero(G, d, dv, n, N):
    """The append form without ACCUMULATE, on states filled with garbage
    first: every head against the oracle, the padding rows come back zero,
    and a second run is bitwise equal."""
    T = G.T
    cfg = T.Config(2, 8, d, dv, n, "bf16")
    assert T.prefill_plan(cfg, N)["ctas_per_sm"] == 3
    q, k, v = G.make_inputs(cfg, N, seed=500 + d + dv + n + N)
    st = T.new_states(cfg, q.device)
    st.fill_(7.0)
    o1, s1 = G.gpu_prefill(cfg, q, k, v, states=st)
    o2, s2 = G.gpu_prefill(cfg, q, k, v, states=st.clone().fill_(-3.0))
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    _check_all_heads(G, cfg, N, seed=500 + d + dv + n + N)
    D, Dp = T.feature_dim(d, n), T.state_pad_dim(d, n)
    sv = s1.view(16, Dp * (dv + 1))
    assert torch.count_nonzero(sv[:, :Dp * dv].view(16, Dp, dv)[:, D:]) == 0
    assert torch.count_nonzero(sv[:, Dp * dv:][:, D:]) == 0


@pytest.mark.parametrize("N", [1, 2, 7, 15, 16, 63])
def test_append_form_short_and_ragged(G, N):
    """chunk = 128 keeps bf16 segments of 1..16 tokens off the short path, so
    the append form runs the smallest segments too (a single token: one key,
    one query row): every head against the oracle, from zero and continuing
    a prefix."""
    T, O = G.T, G.O
    cfg = T.Config(2, 4, 16, 64, 3, "bf16", chunk=128)
    assert T.prefill_plan(cfg, N)["ctas_per_sm"] == 3
    _check_all_heads(G, cfg, N, seed=600 + N)
    P = 129
    q, k, v = G.make_inputs(cfg, P + N, seed=610 + N)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    _, st = G.gpu_prefill(cfg, sl(q, 0, P), sl(k, 0, P), sl(v, 0, P))
    out, st = G.gpu_prefill(cfg, sl(q, P, P + N), sl(k, P, P + N), sl(v, P, P + N), states=st, accumulate=True)
    Sg, og = G.canonical(cfg, st), G.host(out)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for b in range(2):
        for h in range(4):
            o_r, S_r = O.prefill_recurrent(qh[b, h], kh[b, h], vh[b, h], 3)
            G.check_head(cfg, og[b, h], Sg[b, h], o_r[P:], S_r, G.TOL["bf16"], f"append N={N} ({b},{h})")


@pytest.mark.parametrize("d,dv,n,L", [(16, 64, 3, 17), (16, 64, 3, 32), (16, 64, 3, 33), (16, 64, 3, 64),
                                      (32, 64, 2, 50), (16, 32, 1, 64), (16, 32, 3, 40)])
def test_append_many_heads(G, d, dv, n, L):
    """Appends of L tokens with ACCUMULATE to the states of a 300-token
    prefix, on 512 heads (several waves of the append form's three CTAs per
    SM): sampled heads against the oracle run on prefix + segment."""
    T, O = G.T, G.O
    cfg = T.Config(16, 32, d, dv, n, "bf16")
    P = 300
    q, k, v = G.make_inputs(cfg, P + L, seed=70 + d + dv + n + L)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    _, st = G.gpu_prefill(cfg, sl(q, 0, P), sl(k, 0, P), sl(v, 0, P))
    assert T.prefill_plan(cfg, L)["ctas_per_sm"] == 3
    out, st = G.gpu_prefill(cfg, sl(q, P, P + L), sl(k, P, P + L), sl(v, P, P + L), states=st, accumulate=True)
    Sg = G.canonical(cfg, st)
    og = G.host(out)
    for b, h in G.sample_heads(16, 32, k=4, seed=L):
        qh, kh, vh = (G.host(x[b, h]) for x in (q, k, v))
        o_r, S_r = O.prefill_recurrent(qh, kh, vh, n)
        G.check_head(cfg, og[b, h], Sg[b, h], o_r[P:], S_r, G.TOL["bf16"], f"append L={L} ({b},{h})")
