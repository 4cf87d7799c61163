"""Parity of the CUDA path (through the C ABI) with the float64 oracle, on the
same seeded inputs: small cases element by element over every head, and the
full-size workloads on sampled heads (heads are independent, so a sampled head
is checked exactly as it would be alone)."""
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


def _all_heads(G, cfg, N, seed, accumulate_from=None):
    T, O = G.T, G.O
    q, k, v = G.make_inputs(cfg, N, seed)
    out, st = G.gpu_prefill(cfg, q, k, v)
    torch.cuda.synchronize()
    Sg = G.canonical(cfg, st)
    og = G.host(out)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    tol = G.TOL[cfg.dtype]
    errs = []
    for b in range(cfg.B):
        for h in range(cfg.H):
            o_r, S_r = O.prefill_recurrent(qh[b, h], kh[b, h], vh[b, h], cfg.n_terms)
            errs.append(G.check_head(cfg, og[b, h], Sg[b, h], o_r, S_r, tol, f"N={N} b={b} h={h}"))
    return errs


def test_single_head_prefill_then_64_decode_steps(G):
    """B=1 H=1 N=256 d16 dv64 n=3 fp32, seed 0; then 64 decode steps on fresh
    seeded tokens, each compared with the oracle's decode step."""
    T, O = G.T, G.O
    cfg = T.Config(1, 1, 16, 64, 3, "f32")
    q, k, v = G.make_inputs(cfg, 256, seed=0)
    out, st = G.gpu_prefill(cfg, q, k, v)
    o_r, S_r = O.prefill_recurrent(G.host(q)[0, 0], G.host(k)[0, 0], G.host(v)[0, 0], 3)
    G.check_head(cfg, G.host(out)[0, 0], G.canonical(cfg, st)[0, 0], o_r, S_r, 1e-4, "prefill")
    dq, dk, dv = G.make_inputs(cfg, 64, seed=0, phase=1)
    dqh, dkh, dvh = G.host(dq)[0, 0], G.host(dk)[0, 0], G.host(dv)[0, 0]
    o1 = torch.empty((1, 1, 64), dtype=torch.float32, device="cuda")
    S = S_r
    worst = 0.0
    for t in range(64):
        T.decode_step(cfg, dq[:, :, t].contiguous(), dk[:, :, t].contiguous(),
                      dv[:, :, t].contiguous(), o1, st)
        o_ref, S = O.decode_step(dqh[t], dkh[t], dvh[t], S, 3)
        worst = max(worst, G.rel_err(G.host(o1)[0, 0], o_ref))
    assert worst <= 1e-4, worst
    Sg = G.canonical(cfg, st)[0, 0]
    assert G.rel_err(Sg[:, :64], S[:, :64]) <= 1e-4
    assert G.rel_err(Sg[:, 64], S[:, 64]) <= 1e-4


@pytest.mark.parametrize("N", [1, 2, 3, 63, 64, 65, 127, 129, 300, 1000])
def test_ragged_lengths(G, N):
    cfg = G.T.Config(2, 3, 16, 64, 3, "f32")
    _all_heads(G, cfg, N, seed=100 + N)


@pytest.mark.parametrize("N", [1, 2, 31, 32])
def test_ragged_lengths_tensor_core_chunk(G, N):
    """Short sequences forced onto the 128-token tensor-core chunk (the
    library's own choice there is the short-segment prefill)."""
    cfg = G.T.Config(2, 3, 16, 64, 3, "f32", chunk=128)
    assert G.T.prefill_plan(cfg, N)["path"] == G.T.TSA_PATH_TC_F32
    _all_heads(G, cfg, N, seed=150 + N)


@pytest.mark.parametrize("d,dv,n,dtype,N", [
    (16, 64, 3, "f32", 1), (16, 64, 3, "f32", 17), (16, 64, 3, "f32", 32), (16, 64, 3, "f32", 64),
    (16, 64, 3, "f32", 300),     # chunk = 16 asked for: 19 blocks, ragged tail
    (16, 64, 3, "bf16", 40), (16, 32, 3, "f32", 33), (16, 128, 2, "f32", 50),
    (16, 64, 1, "bf16", 20), (32, 128, 2, "f32", 31), (32, 32, 1, "bf16", 5),
])
def test_short_segment_shapes(G, d, dv, n, dtype, N):
    """The short-segment prefill (head state in shared memory, 16-token
    blocks): from zero, and continuing a 100-token prefix with ACCUMULATE."""
    T, O = G.T, G.O
    cfg = T.Config(2, 3, d, dv, n, dtype, chunk=16)
    assert T.prefill_plan(cfg, N)["path"] == T.TSA_PATH_SHORT
    _all_heads(G, cfg, N, seed=400 + N + d + dv + n)
    pre = T.Config(2, 3, d, dv, n, dtype)
    q, k, v = G.make_inputs(cfg, 100 + N, seed=500 + N)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    _, st = G.gpu_prefill(pre, sl(q, 0, 100), sl(k, 0, 100), sl(v, 0, 100))
    out, st = G.gpu_prefill(cfg, sl(q, 100, 100 + N), sl(k, 100, 100 + N), sl(v, 100, 100 + N),
                            states=st, accumulate=True)
    Sg, og = G.canonical(cfg, st), G.host(out)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for b in range(2):
        for h in range(3):
            o_r, S_r = O.prefill_recurrent(qh[b, h], kh[b, h], vh[b, h], n)
            G.check_head(cfg, og[b, h], Sg[b, h], o_r[100:], S_r, G.TOL[dtype], f"append b={b} h={h}")


@pytest.mark.parametrize("d,dv,n,dtype", [
    (16, 64, 1, "f32"), (16, 64, 2, "f32"), (16, 64, 4, "f32"), (32, 128, 3, "f32"),
    (32, 32, 3, "f32"), (16, 32, 4, "f32"), (16, 32, 3, "f32"), (32, 32, 2, "f32"),
    (32, 64, 2, "f32"), (16, 128, 3, "bf16"), (16, 64, 4, "bf16"),
    (32, 128, 3, "bf16"), (32, 64, 2, "bf16"), (16, 64, 3, "bf16"),
])
def test_shapes(G, d, dv, n, dtype):
    cfg = G.T.Config(1, 2, d, dv, n, dtype)
    _all_heads(G, cfg, 333, seed=7 + d + dv + n)


@pytest.mark.parametrize("d,dv,n", [(16, 32, 3), (32, 32, 2), (32, 64, 2), (16, 64, 2)])
def test_fp32_tensor_core_shapes_multi_span(G, d, dv, n):
    """fp32 shapes on the tensor cores (16-column output halves, a 48-row
    last feature block, direct output stores) cut into several spans: the span
    pass, the scan and the bulk-copied span prefixes at other state sizes."""
    cfg = G.T.Config(1, 2, d, dv, n, "f32")
    plan = G.T.prefill_plan(cfg, 3000)
    assert plan["path"] == G.T.TSA_PATH_TC_F32 and plan["n_spans"] > 1, plan
    _all_heads(G, cfg, 3000, seed=50 + d + dv + n)


def test_n1_is_running_mean(G):
    """With one Taylor term every weight is 1: out_i = mean(v_0..v_i)."""
    cfg = G.T.Config(1, 2, 16, 64, 1, "f32")
    q, k, v = G.make_inputs(cfg, 500, seed=3)
    out, _ = G.gpu_prefill(cfg, q, k, v)
    vh = G.host(v)
    want = np.cumsum(vh, axis=2) / np.arange(1, 501)[None, None, :, None]
    assert G.rel_err(G.host(out), want) <= 1e-5


def test_multi_span_8192(G):
    """B=1 H=8 N=8192 d16 dv64 n=3 fp32 (the prefill workload the benchmark
    times, same launch configuration), every head, spans scanned."""
    cfg = G.T.Config(1, 8, 16, 64, 3, "f32")
    assert G.T.prefill_plan(cfg, 8192)["n_spans"] > 1
    _all_heads(G, cfg, 8192, seed=2)


@pytest.mark.parametrize("chunk,path", [(64, 0), (128, 2)])
def test_prefill_8192_chunk_sizes(G, chunk, path):
    """The 8192-token prefill workload at the chunk lengths the library
    builds for fp32: 64 (CUDA cores) and 128 (tensor cores, the default);
    every head."""
    cfg = G.T.Config(1, 8, 16, 64, 3, "f32", chunk)
    plan = G.T.prefill_plan(cfg, 8192)
    assert plan["chunk"] == chunk and plan["path"] == path, plan
    _all_heads(G, cfg, 8192, seed=12 + chunk)


def test_accumulate_continues_the_sequence(G):
    T, O = G.T, G.O
    cfg = T.Config(1, 2, 16, 64, 3, "f32")
    q, k, v = G.make_inputs(cfg, 1200, seed=11)
    _, st = G.gpu_prefill(cfg, q[:, :, :700].contiguous(), k[:, :, :700].contiguous(),
                          v[:, :, :700].contiguous())
    out2, st = G.gpu_prefill(cfg, q[:, :, 700:].contiguous(), k[:, :, 700:].contiguous(),
                             v[:, :, 700:].contiguous(), states=st, accumulate=True)
    Sg = G.canonical(cfg, st)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for h in range(2):
        o_r, S_r = O.prefill_recurrent(qh[0, h], kh[0, h], vh[0, h], 3)
        G.check_head(cfg, G.host(out2)[0, h], Sg[0, h], o_r[700:], S_r, 1e-4, "accumulate")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_short_appends_B64_H16(G, dtype):
    """B=64 H=16 d16 dv64 n=3 (the decode workload's heads): states from a
    300-token prefill, then segments of 1, 16, 64 and 200 tokens appended in
    turn with ACCUMULATE (the launch configuration of the benchmark's short
    appends); sampled heads checked segment by segment against the oracle
    continuing from its own state."""
    T = G.T
    cfg = T.Config(64, 16, 16, 64, 3, dtype)
    tol = G.TOL[dtype]
    q, k, v = G.make_inputs(cfg, 300, seed=21)
    _, st = G.gpu_prefill(cfg, q, k, v)
    heads = G.sample_heads(64, 16, k=2, seed=21)
    S_refs = {}
    for (b, h) in heads:
        _, S_refs[(b, h)] = G.oracle_prefill(G.host(q[b, h]), G.host(k[b, h]), G.host(v[b, h]), 3)
    for phase, L in enumerate((1, 16, 64, 200), start=1):
        aq, ak, av = G.make_inputs(cfg, L, seed=21, phase=phase)
        out, st = G.gpu_prefill(cfg, aq, ak, av, states=st, accumulate=True)
        Sg = G.canonical(cfg, st)
        og = G.host(out)
        for (b, h) in heads:
            o_r, S_r = G.oracle_prefill(G.host(aq[b, h]), G.host(ak[b, h]), G.host(av[b, h]), 3,
                                        S0=S_refs[(b, h)])
            G.check_head(cfg, og[b, h], Sg[b, h], o_r, S_r, tol, f"L={L} head {(b, h)}")
            S_refs[(b, h)] = S_r


@pytest.mark.parametrize("d,dtype", [(16, "f32"), (32, "f32"), (16, "bf16")])
def test_order_sweep_against_softmax(G, d, dtype):
    """Accuracy against exact causal softmax as the number of Taylor terms
    grows, at the state size each order costs (abstract: accuracy improves
    quickly with n while the state widens combinatorially). On the same
    inputs the CUDA path's error against softmax equals the oracle's own
    truncation error to within the parity tolerance, and it falls strictly
    from one order to the next."""
    T, O = G.T, G.O
    orders = [1, 2, 3, 4, 5] if d == 16 else [1, 2, 3]
    B, H, N, dv = 1, 4, 512, 64
    errs = []
    for n in orders:
        cfg = T.Config(B, H, d, dv, n, dtype)
        q, k, v = G.make_inputs(cfg, N, seed=60 + d)
        out, _ = G.gpu_prefill(cfg, q, k, v)
        og, qh, kh, vh = G.host(out), G.host(q), G.host(k), G.host(v)
        e_gpu = e_ref = 0.0
        for h in range(H):
            sm = O.softmax_attention(qh[0, h], kh[0, h], vh[0, h])
            ref = O.attention_direct(qh[0, h], kh[0, h], vh[0, h], n)
            e_gpu = max(e_gpu, G.rel_err(og[0, h], sm))
            e_ref = max(e_ref, G.rel_err(ref, sm))
        assert abs(e_gpu - e_ref) <= G.TOL[dtype], (n, e_gpu, e_ref)
        errs.append((T.state_elems(cfg), e_gpu, e_ref))
    # the truncation error falls with every order; the GPU's error with it
    # wherever the drop exceeds twice the rounding of the output dtype (bf16:
    # 2^-8; from n = 4 to 5 the drop, ~2e-3, is below that in bf16)
    noise = 2.0 ** -8 if dtype == "bf16" else 0.0
    for (s0, e0, r0), (s1, e1, r1) in zip(errs, errs[1:]):
        assert s1 > s0 and r1 < r0, errs
        if r0 - r1 > 2 * noise:
            assert e1 < e0, errs


def test_merge_of_segments_equals_whole(G):
    T, O = G.T, G.O
    cfg = T.Config(2, 2, 16, 64, 3, "f32")
    q, k, v = G.make_inputs(cfg, 900, seed=12)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    _, sa = G.gpu_prefill(cfg, sl(q, 0, 400), sl(k, 0, 400), sl(v, 0, 400))
    _, sb = G.gpu_prefill(cfg, sl(q, 400, 900), sl(k, 400, 900), sl(v, 400, 900))
    T.state_merge(cfg, sa, sb)
    Sg = G.canonical(cfg, sa)
    kh, vh = G.host(k), G.host(v)
    for b in range(2):
        for h in range(2):
            S_r = sum(O.chunk_states(kh[b, h], vh[b, h], 3, 900))
            assert G.rel_err(Sg[b, h][:, :64], S_r[:, :64]) <= 1e-4
            assert G.rel_err(Sg[b, h][:, 64], S_r[:, 64]) <= 1e-4


def test_decode_equals_next_prefill_row(G):
    T, O = G.T, G.O
    cfg = T.Config(1, 4, 16, 64, 3, "f32")
    q, k, v = G.make_inputs(cfg, 513, seed=13)
    _, st = G.gpu_prefill(cfg, q[:, :, :512].contiguous(), k[:, :, :512].contiguous(),
                          v[:, :, :512].contiguous())
    o1 = torch.empty((1, 4, 64), dtype=torch.float32, device="cuda")
    T.decode_step(cfg, q[:, :, 512].contiguous(), k[:, :, 512].contiguous(),
                  v[:, :, 512].contiguous(), o1, st)
    full, st_full = G.gpu_prefill(cfg, q, k, v)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for h in range(4):
        o_r, S_r = O.prefill_recurrent(qh[0, h], kh[0, h], vh[0, h], 3)
        assert G.rel_err(G.host(o1)[0, h], o_r[512]) <= 1e-4
        assert G.rel_err(G.host(full)[0, h, 512], o_r[512]) <= 1e-4
    assert G.rel_err(G.canonical(cfg, st), G.canonical(cfg, st_full)) <= 1e-5


def test_deterministic_and_padding_zero(G):
    T = G.T
    cfg = T.Config(1, 8, 16, 64, 3, "f32")
    q, k, v = G.make_inputs(cfg, 3000, seed=14)
    o1, s1 = G.gpu_prefill(cfg, q, k, v)
    o2, s2 = G.gpu_prefill(cfg, q, k, v)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    D, Dp = T.feature_dim(16, 3), T.state_pad_dim(16, 3)
    st = s1.view(8, Dp * 65)
    S = st[:, :Dp * 64].view(8, Dp, 64)
    z = st[:, Dp * 64:]
    assert torch.count_nonzero(S[:, D:]) == 0 and torch.count_nonzero(z[:, D:]) == 0


def test_empty_sequence(G):
    T = G.T
    cfg = T.Config(1, 2, 16, 64, 3, "f32")
    st = torch.randn(T.state_bytes(cfg) // 4, device="cuda")
    keep = st.clone()
    e = torch.empty(0, device="cuda")
    q = torch.empty((1, 2, 0, 16), device="cuda")
    T.prefill(cfg, 0, q, q, q, q, st, accumulate=True)
    assert torch.equal(st, keep)
    T.prefill(cfg, 0, q, q, q, q, st, accumulate=False)
    assert torch.count_nonzero(st) == 0
    del e


# ---------------------------------------------------------------------------
# full-size workloads, sampled heads
# ---------------------------------------------------------------------------

def _sampled_prefill_check(G, cfg, q, k, v, out, st, heads, chunked=256):
    O = G.O
    tol = G.TOL[cfg.dtype]
    Sg = T_canon = G.canonical(cfg, st)
    S_refs = {}
    for (b, h) in heads:
        qh, kh, vh = G.host(q[b, h]), G.host(k[b, h]), G.host(v[b, h])
        o_r, S_r = G.oracle_prefill(qh, kh, vh, cfg.n_terms, chunked=chunked)
        G.check_head(cfg, G.host(out[b, h]), Sg[b, h], o_r, S_r, tol, f"head {(b, h)}")
        S_refs[(b, h)] = S_r
    del T_canon
    return S_refs


def _decode_steps_check(G, cfg, st, S_refs, steps, seed):
    """Run `steps` decode steps for all heads on the GPU; compare the sampled
    heads' outputs at every step with the oracle's decode from its own state."""
    T, O = G.T, G.O
    dq, dk, dv = G.make_inputs(cfg, steps, seed=seed, phase=1)
    outs = torch.empty((steps, cfg.B, cfg.H, cfg.d_v), dtype=dq.dtype, device="cuda")
    qs = dq.permute(2, 0, 1, 3).contiguous()
    ks = dk.permute(2, 0, 1, 3).contiguous()
    vs = dv.permute(2, 0, 1, 3).contiguous()
    for t in range(steps):
        T.decode_step(cfg, qs[t], ks[t], vs[t], outs[t], st)
    torch.cuda.synchronize()
    tol = G.TOL[cfg.dtype]
    Sg = G.canonical(cfg, st)
    for (b, h), S in S_refs.items():
        qh, kh, vh = G.host(qs[:, b, h]), G.host(ks[:, b, h]), G.host(vs[:, b, h])
        og = G.host(outs[:, b, h])
        worst = 0.0
        for t in range(steps):
            o_ref, S = O.decode_step(qh[t], kh[t], vh[t], S, cfg.n_terms)
            worst = max(worst, G.rel_err(og[t], o_ref))
        assert worst <= tol, (b, h, worst)
        assert G.rel_err(Sg[b, h][:, :cfg.d_v], S[:, :cfg.d_v]) <= tol
        assert G.rel_err(Sg[b, h][:, cfg.d_v], S[:, cfg.d_v]) <= tol


def test_full_decode_B64_H16_N65536(G):
    """B=64 H=16 d16 dv64 n=3 bf16: prefill of 65,536 tokens, then 1024 decode
    steps (the decode workload the benchmark times)."""
    T = G.T
    cfg = T.Config(64, 16, 16, 64, 3, "bf16")
    q, k, v = G.make_inputs(cfg, 65536, seed=3)
    out, st = G.gpu_prefill(cfg, q, k, v)
    heads = G.sample_heads(64, 16, k=2, seed=3)
    S_refs = _sampled_prefill_check(G, cfg, q, k, v, out, st, heads)
    del q, k, v, out
    torch.cuda.empty_cache()
    _decode_steps_check(G, cfg, st, S_refs, 1024, seed=3)


def test_full_order4_B4_H16_N32768(G):
    T = G.T
    cfg = T.Config(4, 16, 16, 64, 4, "bf16")
    q, k, v = G.make_inputs(cfg, 32768, seed=4)
    out, st = G.gpu_prefill(cfg, q, k, v)
    heads = G.sample_heads(4, 16, k=2, seed=4)
    S_refs = _sampled_prefill_check(G, cfg, q, k, v, out, st, heads)
    del q, k, v, out
    _decode_steps_check(G, cfg, st, S_refs, 256, seed=4)


def test_full_wide_B2_H32_N65536_with_merge(G):
    T, O = G.T, G.O
    cfg = T.Config(2, 32, 32, 128, 3, "bf16")
    q, k, v = G.make_inputs(cfg, 65536, seed=5)
    out, st = G.gpu_prefill(cfg, q, k, v)
    heads = G.sample_heads(2, 32, k=2, seed=5)
    S_refs = _sampled_prefill_check(G, cfg, q, k, v, out, st, heads)
    # merge check: prefill of the two halves, states summed, vs the whole
    half = 32768
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    _, sa = G.gpu_prefill(cfg, sl(q, 0, half), sl(k, 0, half), sl(v, 0, half))
    _, sb = G.gpu_prefill(cfg, sl(q, half, 65536), sl(k, half, 65536), sl(v, half, 65536))
    T.state_merge(cfg, sa, sb)
    Sm = G.canonical(cfg, sa)
    for (b, h), S_r in S_refs.items():
        assert G.rel_err(Sm[b, h][:, :128], S_r[:, :128]) <= G.TOL["bf16"]
        assert G.rel_err(Sm[b, h][:, 128], S_r[:, 128]) <= G.TOL["bf16"]
    # and the merged state agrees with the single-pass state on every head
    assert G.rel_err(G.host(sa), G.host(st)) <= 1e-4


def test_more_heads_than_a_grid_y_dimension(G):
    """70,000 heads (beyond the 65,535 blocks a grid's y dimension allows):
    the state-only prefill (span pass and scan), the prefill and a decode
    step all cover every head; the two prefills give the same states, and
    sampled heads match the oracle."""
    T, O = G.T, G.O
    cfg = T.Config(70, 1000, 16, 32, 1, "f32")
    N = 5
    q, k, v = G.make_inputs(cfg, N + 1, seed=77)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    s1 = T.new_states(cfg)
    T.prefill_states(cfg, N, sl(k, 0, N), sl(v, 0, N), s1)
    out, s2 = G.gpu_prefill(cfg, sl(q, 0, N), sl(k, 0, N), sl(v, 0, N))
    T.sync_status()
    # (the state-only call takes the split-bf16 tensor cores, the prefill the
    # CUDA cores: equal up to the fp32 parity tolerance)
    assert G.rel_err(G.host(s1), G.host(s2)) <= G.TOL["f32"]
    od = torch.empty((70, 1000, 32), device="cuda")
    T.decode_step(cfg, q[:, :, N].contiguous(), k[:, :, N].contiguous(), v[:, :, N].contiguous(), od, s2)
    T.sync_status()
    Sg, og, odh = G.canonical(cfg, s2), G.host(out), G.host(od)
    for b, h in [(0, 0), (69, 999), (35, 512), (65, 535)]:
        qh, kh, vh = (G.host(x[b, h]) for x in (q, k, v))
        o_r, S_r = O.prefill_recurrent(qh, kh, vh, 1)
        G.check_head(cfg, og[b, h], Sg[b, h], o_r[:N], S_r, G.TOL["f32"], f"head ({b},{h})")
        assert G.rel_err(odh[b, h], o_r[N]) <= G.TOL["f32"], (b, h)
