"""Small-shape parity of every path with the library's debug build
(libtsa_debug.so: device-side checks before each TMEM, shared-memory operand,
TMA and state access).

Run as a child process with TSA_DEBUG=1 in its environment (the binding picks
the library when it is imported), from tests/test_gpu_debug_build.py:
    TSA_DEBUG=1 python tests/debug_build_cases.py
Every case runs one call, asks tsa_sync_status for the device checks (any
failed check is TSA_ERR_DEVICE_CHECK) and compares with the float64 oracle.
The first case makes a check fail on purpose (the self-test: a TMEM column
check on columns past the allocation, with no access made) and expects the
report. Prints one line per case and "debug build ok" at the end."""
from __future__ import annotations

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import gpu_helpers as G  # noqa: E402

T, O = G.T, G.O


def selftest():
    assert T.debug_build(), "the debug build was not loaded"
    T.sync_status()
    T.debug_check_selftest()
    try:
        T.sync_status()
    except T.TsaError as e:
        assert e.status == T.TSA_ERR_DEVICE_CHECK, e
        assert "TMEM columns" in str(e) and "(510, 16)" in str(e), e
        print("selftest:", e)
    else:
        raise AssertionError("the failed check was not reported")
    T.sync_status()   # the report was cleared


def prefill_case(d, dv, n, dtype, N, H=2, chunk=0, expect_path=None, expect_cluster=None, accumulate_pre=0):
    cfg = T.Config(1, H, d, dv, n, dtype, chunk)
    plan = T.prefill_plan(cfg, N)
    if expect_path is not None:
        assert plan["path"] == expect_path, plan
    if expect_cluster is not None:
        assert plan["cluster"] == expect_cluster, plan
    q, k, v = G.make_inputs(cfg, accumulate_pre + N, seed=900 + d + dv + n + N)
    seg = lambda x, a, b: x[:, :, a:b].contiguous()
    st = None
    if accumulate_pre:
        _, st = G.gpu_prefill(cfg, seg(q, 0, accumulate_pre), seg(k, 0, accumulate_pre), seg(v, 0, accumulate_pre))
    out, st = G.gpu_prefill(cfg, seg(q, accumulate_pre, accumulate_pre + N), seg(k, accumulate_pre, accumulate_pre + N),
                            seg(v, accumulate_pre, accumulate_pre + N), states=st, accumulate=bool(accumulate_pre))
    S = G.canonical(cfg, st)
    qh, kh, vh, og = G.host(q), G.host(k), G.host(v), G.host(out)
    worst = 0.0
    for h in range(H):
        o_r, S_r = G.oracle_prefill(qh[0, h], kh[0, h], vh[0, h], n, chunked=128 if N > 2000 else None)
        e = G.check_head(cfg, og[0, h], S[0, h], o_r[accumulate_pre:], S_r, G.TOL[dtype], f"head {h}")
        worst = max(worst, *e)
    print(f"prefill d{d} dv{dv} n{n} {dtype} N={N} chunk={chunk} pre={accumulate_pre} path={plan['path']} "
          f"cluster={plan['cluster']} spans={plan['n_spans']}: worst {worst:.2e}")


def decode_merge_states_case():
    cfg = T.Config(2, 2, 16, 64, 3, "bf16")
    N = 150
    q, k, v = G.make_inputs(cfg, N + 1, seed=77)
    seg = lambda x, a, b: x[:, :, a:b].contiguous()
    _, st = G.gpu_prefill(cfg, seg(q, 0, N), seg(k, 0, N), seg(v, 0, N))
    o1 = torch.empty((2, 2, 64), dtype=q.dtype, device="cuda")
    T.decode_step(cfg, q[:, :, N].contiguous(), k[:, :, N].contiguous(), v[:, :, N].contiguous(), o1, st)
    T.sync_status()
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for b in range(2):
        for h in range(2):
            o_r, _ = O.prefill_recurrent(qh[b, h], kh[b, h], vh[b, h], 3)
            assert G.rel_err(G.host(o1[b, h]), o_r[N]) <= G.TOL["bf16"], (b, h)
    # merge: the sums of two halves equal the state of the whole
    a = T.new_states(cfg)
    T.prefill_states(cfg, 70, seg(k, 0, 70), seg(v, 0, 70), a)
    bst = T.new_states(cfg)
    T.prefill_states(cfg, N + 1 - 70, seg(k, 70, N + 1), seg(v, 70, N + 1), bst)
    T.state_merge(cfg, a, bst)
    T.sync_status()
    S = G.canonical(cfg, a)
    Sw = G.canonical(cfg, st)
    assert G.rel_err(S[..., :64], Sw[..., :64]) <= G.TOL["bf16"]
    print("decode, prefill_states, merge: ok")


def feature_map_case():
    x = torch.randn((300, 16), device="cuda")
    x = x / torch.linalg.vector_norm(x, dim=1, keepdim=True)
    D = T.feature_dim(16, 3)
    phi = torch.empty((300, D), device="cuda")
    T.feature_map(16, 3, x, phi)
    T.sync_status()
    assert np.abs(G.host(phi) - O.phi(G.host(x), 3)).max() <= 1e-6
    print("feature_map: ok")


def main():
    selftest()
    prefill_case(16, 64, 3, "bf16", 300, expect_path=T.TSA_PATH_TC, expect_cluster=1)
    prefill_case(16, 64, 4, "bf16", 700, expect_path=T.TSA_PATH_TC, expect_cluster=2)
    prefill_case(32, 128, 3, "bf16", 260, expect_path=T.TSA_PATH_TC, expect_cluster=2)
    prefill_case(16, 64, 3, "f32", 1000, expect_path=T.TSA_PATH_TC_F32)
    prefill_case(16, 64, 3, "f32", 8192, H=2, expect_path=T.TSA_PATH_TC_F32)   # several spans, the scan
    prefill_case(16, 64, 3, "f32", 500, chunk=64, expect_path=T.TSA_PATH_SIMT)
    prefill_case(16, 64, 3, "f32", 16, expect_path=T.TSA_PATH_SHORT, accumulate_pre=40)
    prefill_case(16, 64, 3, "bf16", 200, accumulate_pre=129)
    prefill_case(16, 64, 3, "bf16", 50, H=4, accumulate_pre=100)   # the append form, two feature blocks
    prefill_case(16, 32, 1, "bf16", 64, H=4, accumulate_pre=100)   # append form, the smallest state
    prefill_case(32, 64, 2, "bf16", 40, H=4, accumulate_pre=100)   # append form, d_k 32
    prefill_case(16, 64, 3, "bf16", 24, H=4)                       # append form from a zero state
    prefill_case(16, 64, 3, "bf16", 1, H=4, chunk=128, accumulate_pre=129)   # append form, one token
    prefill_case(16, 64, 4, "f32", 300, expect_path=T.TSA_PATH_SIMT)          # one 64-column slice, global state
    prefill_case(16, 64, 5, "f32", 200, expect_path=T.TSA_PATH_SIMT, accumulate_pre=70)   # n = 5, several spans
    decode_merge_states_case()
    feature_map_case()
    print("debug build ok")


if __name__ == "__main__":
    main()
