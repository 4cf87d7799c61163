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
    cases = [
        (T.Config(1, 8, 16, 64, 3, "f32"), 8192, 21, 1e-4),    # 32 spans: scratch in use
        (T.Config(1, 2, 32, 128, 3, "bf16"), 3000, 22, 2e-2),   # 24 spans, 13.3 MiB
    ]
    for cfg, N, seed, tol in cases:
        plan = T.prefill_plan(cfg, N)
        assert plan["scratch_bytes"] > 0 and plan["scratch_bytes"] <= 16 << 20
        q, k, v = torch_qkv(cfg.B, cfg.H, N, cfg.d_k, cfg.d_v, cfg.dtype, seed, device="cuda")
        ref_out = torch.empty((cfg.B, cfg.H, N, cfg.d_v), dtype=q.dtype, device="cuda")
        ref_st = T.new_states(cfg)
        T.prefill(cfg, N, q, k, v, ref_out, ref_st)
        for call in range(2):
            out = torch.full_like(ref_out, float("nan"))
            st = T.new_states(cfg)
            T.prefill_noalloc(cfg, N, q, k, v, out, st)
            torch.cuda.synchronize()
            for b in range(cfg.B):
                for h in range(cfg.H):
                    assert _rel(out[b, h], ref_out[b, h]) <= tol, (cfg, call, b, h)
            assert _rel(st, ref_st) <= tol, (cfg, call)


def test_noalloc_refuses_oversize_plan(T):
    cfg = T.Config(1, 16, 32, 128, 3, "bf16")
    N = 65536
    plan = T.prefill_plan(cfg, N)
    if plan["scratch_bytes"] <= 16 << 20:
        pytest.skip("this device's plan fits the static buffer")
    q = torch.zeros((1, 16, N, 32), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, 16, N, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(v, 7.0)
    st = T.new_states(cfg)
    with pytest.raises(T.TsaError) as e:
        T.prefill_noalloc(cfg, N, q, q, v, out, st)
    assert e.value.status == T.TSA_ERR_UNSUPPORTED
    assert "static buffer" in T.last_error()
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
