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


def test_noalloc_refuses_oversize_plan(T):
    # 64 fp32 heads of 65,536 tokens: the plan spreads each head over several
    # spans, whose states need about 40 MiB of scratch on a 148-SM part
    cfg = T.Config(1, 64, 16, 64, 3, "f32")
    N = 65536
    plan = T.prefill_plan(cfg, N)
    assert plan["scratch_bytes"] > 16 << 20, plan
    q = torch.zeros((1, 64, N, 16), dtype=torch.float32, device="cuda")
    v = torch.zeros((1, 64, N, 64), dtype=torch.float32, device="cuda")
    out = torch.full_like(v, 7.0)
    st = T.new_states(cfg)
    with pytest.raises(T.TsaError) as e:
        T.prefill_noalloc(cfg, N, q, q, v, out, st)
    assert e.value.status == T.TSA_ERR_UNSUPPORTED
    assert "static buffer" in T.last_error()
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
