"""Failure detection on the GPU without a fault: a bounded device-side wait
that runs out is reported as TSA_ERR_TIMEOUT, and the context stays usable.

The testing hooks of the library shorten the bound of every wait between the
warp roles of the tensor-core kernels to a few milliseconds and make the fp32
output pass withhold one publication (the first chunk's completed output
accumulator), so the warps waiting for it give up: each CTA sets its abort
flag, stops issuing work, waits (bounded) for what it has in flight, releases
its tensor memory and exits, and records the failure in the library's device
error word. tsa_sync_status must then report TSA_ERR_TIMEOUT once; a normal
prefill in the same process must afterwards match the oracle (its CTAs
allocate the tensor memory the aborted ones released).
"""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrence_phi_b300 import build
    build.build()
    from fixed_state_recurrence_phi_b300 import tsa
    return tsa


def test_withheld_publication_times_out_then_prefill_is_correct(T):
    from gpu_helpers import check_head, host, make_inputs, oracle_prefill, canonical, TOL
    cfg = T.Config(1, 2, 16, 64, 3, "f32")
    N = 700
    assert T.prefill_plan(cfg, N)["path"] == T.TSA_PATH_TC_F32
    q, k, v = make_inputs(cfg, N, seed=31)
    out = torch.zeros((1, 2, N, 64), device="cuda")
    st = T.new_states(cfg)
    T.sync_status()
    T.debug_set_wait_limit(2_000_000)          # 2 ms per wait
    T.debug_withhold_publication(1)
    try:
        T.prefill(cfg, N, q, k, v, out, st)
        with pytest.raises(T.TsaError) as e:
            T.sync_status()
        assert e.value.status == T.TSA_ERR_TIMEOUT, T.last_error()
    finally:
        T.debug_withhold_publication(0)
        T.debug_set_wait_limit(0)
    T.sync_status()                              # reported once, then cleared
    # the same call again, hooks off: complete and correct
    out.zero_()
    st.zero_()
    T.prefill(cfg, N, q, k, v, out, st)
    T.sync_status()
    S = canonical(cfg, st)
    qh, kh, vh = host(q), host(k), host(v)
    for h in range(2):
        o_r, S_r = oracle_prefill(qh[0, h], kh[0, h], vh[0, h], 3)
        check_head(cfg, host(out[0, h]), S[0, h], o_r, S_r, TOL["f32"], f"head {h}")


def test_pair_exchange_withheld_times_out_then_prefill_is_correct(T):
    """The CTA-pair prefill (bf16, order 4): rank 0 of each pair withholds its
    first partial-output publication to its peer. The peer's bounded wait runs
    out, it passes the abort to rank 0, both release their tensor memory and
    leave through the cluster barrier, and TSA_ERR_TIMEOUT is reported; the
    same prefill afterwards matches the oracle."""
    from gpu_helpers import check_head, host, make_inputs, oracle_prefill, canonical, TOL
    cfg = T.Config(1, 2, 16, 64, 4, "bf16")
    N = 700
    assert T.prefill_plan(cfg, N)["cluster"] == 2
    q, k, v = make_inputs(cfg, N, seed=32)
    out = torch.zeros((1, 2, N, 64), dtype=torch.bfloat16, device="cuda")
    st = T.new_states(cfg)
    T.sync_status()
    T.debug_set_wait_limit(2_000_000)
    T.debug_withhold_publication(2)
    try:
        T.prefill(cfg, N, q, k, v, out, st)
        with pytest.raises(T.TsaError) as e:
            T.sync_status()
        assert e.value.status == T.TSA_ERR_TIMEOUT, T.last_error()
    finally:
        T.debug_withhold_publication(0)
        T.debug_set_wait_limit(0)
    T.sync_status()
    out.zero_()
    st.zero_()
    T.prefill(cfg, N, q, k, v, out, st)
    T.sync_status()
    S = canonical(cfg, st)
    qh, kh, vh = host(q), host(k), host(v)
    for h in range(2):
        o_r, S_r = oracle_prefill(qh[0, h], kh[0, h], vh[0, h], 4)
        check_head(cfg, host(out[0, h]), S[0, h], o_r, S_r, TOL["bf16"], f"head {h}")


def test_append_form_withheld_times_out_then_append_is_correct(T):
    """The bf16 append form (three CTAs per SM, 64-token segments): the issuer
    never publishes that O is complete, the workers' bounded wait runs out,
    every CTA gives up and releases its tensor memory, TSA_ERR_TIMEOUT is
    reported; the same append afterwards, continuing a prefix, matches the
    oracle."""
    from gpu_helpers import check_head, host, make_inputs, canonical, gpu_prefill, TOL
    from oracle import tsa_oracle as O
    cfg = T.Config(2, 8, 16, 64, 3, "bf16")
    P, L = 150, 40
    assert T.prefill_plan(cfg, L)["ctas_per_sm"] == 3
    q, k, v = make_inputs(cfg, P + L, seed=33)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    _, st0 = gpu_prefill(cfg, sl(q, 0, P), sl(k, 0, P), sl(v, 0, P))
    aq, ak, av = sl(q, P, P + L), sl(k, P, P + L), sl(v, P, P + L)
    out = torch.zeros((2, 8, L, 64), dtype=torch.bfloat16, device="cuda")
    st = st0.clone()
    T.sync_status()
    T.debug_set_wait_limit(2_000_000)
    T.debug_withhold_publication(3)
    try:
        T.prefill(cfg, L, aq, ak, av, out, st, accumulate=True)
        with pytest.raises(T.TsaError) as e:
            T.sync_status()
        assert e.value.status == T.TSA_ERR_TIMEOUT, T.last_error()
    finally:
        T.debug_withhold_publication(0)
        T.debug_set_wait_limit(0)
    T.sync_status()
    st = st0.clone()
    T.prefill(cfg, L, aq, ak, av, out, st, accumulate=True)
    T.sync_status()
    S = canonical(cfg, st)
    qh, kh, vh = host(q), host(k), host(v)
    for b, h in [(0, 0), (1, 7), (0, 5)]:
        o_r, S_r = O.prefill_recurrent(qh[b, h], kh[b, h], vh[b, h], 3)
        check_head(cfg, host(out[b, h]), S[b, h], o_r[P:], S_r, TOL["bf16"], f"head ({b},{h})")
