"""tsa_prefill_noalloc: the prefill for callers that cannot allocate device
memory (their memory budget belongs to their own allocator, they must not
allocate once serving, or their GPU lacks the stream-ordered allocator). It
uses one fixed 16 MiB device array instead of pool scratch. Here it is called
through the C ABI twice in a row and checked against tsa_prefill on the same
inputs, with the tolerance of the other parity tests; and a shape needing more
scratch than the array holds is refused before any work is queued.

This file is named to be collected last."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def T():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrence_phi_b300 import build
    build.build()
    from fixed_state_recurrence_phi_b300 import tsa
    return tsa


def _rel(a, b):
    a = a.double().cpu().numpy(); b = b.double().cpu().numpy()
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def test_noalloc_matches_prefill_on_two_calls(T):
    from fixed_state_recurrence_phi_b300.inputs import torch_qkv
    # (config, N, seed, tolerance, continue from existing states); on a 148-SM
    # B300 the plans take 16 spans (5.0 MiB of scratch), 24 spans (13.3 MiB),
    # 16 spans with the caller's states as the scan's start (5.0 MiB), and 63
    # spans of the CUDA-core kernels (chunk 64, 9.7 MiB)
    cases = [
        (T.Config(1, 8, 16, 64, 3, "f32"), 8192, 21, 1e-4, False),
        (T.Config(1, 2, 32, 128, 3, "bf16"), 3000, 22, 2e-2, False),
        (T.Config(1, 8, 16, 64, 3, "bf16"), 8192, 23, 2e-2, True),
        (T.Config(1, 4, 16, 64, 3, "f32", 64), 4000, 24, 1e-4, False),
    ]
    for cfg, N, seed, tol, acc in cases:
        plan = T.prefill_plan(cfg, N)
        assert plan["scratch_bytes"] > 0 and plan["scratch_bytes"] <= 16 << 20
        q, k, v = torch_qkv(cfg.B, cfg.H, N, cfg.d_k, cfg.d_v, cfg.dtype, seed, device="cuda")
        st0 = T.new_states(cfg)
        if acc:   # a prefix of 300 tokens first: its states are the start
            q0, k0, v0 = torch_qkv(cfg.B, cfg.H, 300, cfg.d_k, cfg.d_v, cfg.dtype, seed + 100, device="cuda")
            T.prefill(cfg, 300, q0, k0, v0, torch.empty_like(v0), st0)
        ref_out = torch.empty((cfg.B, cfg.H, N, cfg.d_v), dtype=q.dtype, device="cuda")
        ref_st = st0.clone()
        T.prefill(cfg, N, q, k, v, ref_out, ref_st, accumulate=acc)
        for call in range(2):
            out = torch.full_like(ref_out, float("nan"))
            st = st0.clone()
            T.prefill_noalloc(cfg, N, q, k, v, out, st, accumulate=acc)
            torch.cuda.synchronize()
            for b in range(cfg.B):
                for h in range(cfg.H):
                    assert _rel(out[b, h], ref_out[b, h]) <= tol, (cfg, call, b, h)
            assert _rel(st, ref_st) <= tol, (cfg, call)


def test_noalloc_caps_its_plan_at_the_static_scratch(T):
    # 2 bf16 heads of order 4 and 65,536 tokens: tsa_prefill's plan spreads
    # each head over spans whose states need about 17.8 MiB of scratch, more
    # than the no-alloc array holds; the no-alloc call takes fewer spans and
    # gives the same results (up to the rounding order of the span sums)
    cfg = T.Config(1, 2, 16, 64, 4, "bf16")
    N = 65536
    plan = T.prefill_plan(cfg, N)
    assert plan["scratch_bytes"] > 16 << 20, plan
    from fixed_state_recurrence_phi_b300.inputs import torch_qkv
    q, k, v = torch_qkv(1, 2, N, 16, 64, "bf16", seed=91, device="cuda")
    out_a = torch.empty_like(v)
    out_b = torch.empty_like(v)
    st_a, st_b = T.new_states(cfg), T.new_states(cfg)
    T.prefill(cfg, N, q, k, v, out_a, st_a)
    T.prefill_noalloc(cfg, N, q, k, v, out_b, st_b)
    T.sync_status()
    assert _rel(out_b, out_a) <= 2e-2
    assert _rel(st_b, st_a) <= 1e-4


def test_noalloc_order5_in_place(T):
    """n = 5 (4,845 features, 1.26 MB of state per head): tsa_prefill's plan
    takes several spans whose slots need far more than the 16 MiB array, so
    the no-alloc call plans fewer (down to one span, whose CTA updates the
    caller's state in place) and must give the same results, from zero and
    continuing a prefix."""
    from fixed_state_recurrence_phi_b300.inputs import torch_qkv
    cfg = T.Config(1, 8, 16, 64, 5, "f32")
    N = 640
    assert T.prefill_plan(cfg, N)["scratch_bytes"] > 16 << 20
    q, k, v = torch_qkv(1, 8, N, 16, 64, "f32", 31, device="cuda")
    for acc in (False, True):
        st0 = T.new_states(cfg)
        if acc:
            q0, k0, v0 = torch_qkv(1, 8, 100, 16, 64, "f32", 32, device="cuda")
            T.prefill(cfg, 100, q0, k0, v0, torch.empty_like(v0), st0)
        ref_out = torch.empty((1, 8, N, 64), device="cuda")
        ref_st = st0.clone()
        T.prefill(cfg, N, q, k, v, ref_out, ref_st, accumulate=acc)
        out = torch.full_like(ref_out, float("nan"))
        st = st0.clone()
        T.prefill_noalloc(cfg, N, q, k, v, out, st, accumulate=acc)
        T.sync_status()
        for h in range(8):
            assert _rel(out[0, h], ref_out[0, h]) <= 1e-4, (acc, h)
        assert _rel(st, ref_st) <= 1e-4, acc
