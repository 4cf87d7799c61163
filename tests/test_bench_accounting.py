"""The benchmark's roofline accounting: algorithmic bytes and flops per
workload, against figures worked out by hand from the method's sizes (the
state of d = 16, d_v = 64, n = 3 is 153 x 65 = 9,945 fp32 elements per head,
the abstract's figure; D = 969 at d = 16, n = 4 and 561 at d = 32, n = 3).
No GPU is used."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_accounting", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_prefill_bytes_8192_tokens():
    b = _bench()
    # 8 heads x 8192 tokens x (q 16 + k 16 + v 64 + out 64) fp32, plus the
    # final states 8 x 9,945 fp32
    want = 8 * 8192 * 160 * 4 + 8 * 9945 * 4
    assert want == 42_261_280
    assert b._algorithmic_prefill_bytes(b.PREFILL) == want


def test_decode_and_append_bytes():
    b = _bench()
    # 1,024 heads: the state read and written (2 x 9,945 fp32) plus one
    # token's q, k, v, out in bf16 (160 values)
    assert b._algorithmic_decode_bytes(b.DECODE) == 1024 * (2 * 9945 * 4 + 160 * 2) == 81_797_120
    # a 16-token append: the same state traffic, 16 tokens of bf16 I/O
    assert b._algorithmic_append_bytes(b.DECODE, 16) == 1024 * (2 * 9945 * 4 + 16 * 160 * 2) == 86_712_320


def test_tensor_core_flops():
    b = _bench()
    # per token-head: update and readout 2 x 2*D*(d_v+1), intra-chunk
    # 2*64*(d+d_v+1) at the reference chunk of 64
    order4 = (4 * 969 * 65 + 2 * 64 * (16 + 64 + 1)) * 4 * 16 * 32768
    wide = (4 * 561 * 129 + 2 * 64 * (32 + 128 + 1)) * 2 * 32 * 65536
    assert order4 == 550_099_746_816 and wide == 1_300_586_561_536
    assert b._algorithmic_prefill_flops(b.ORDER4) == order4
    assert b._algorithmic_prefill_flops(b.WIDE) == wide


def test_parity_figures():
    """The bench's parity figures: normwise max|g-r|/max|r| and elementwise
    |g-r|/|r| over the elements with |r| >= 1% of max|r|, worked by hand."""
    import numpy as np
    b = _bench()
    dv = 2
    o_r = np.array([[1.0, -2.0], [0.5, 0.001]])          # 0.001 is under 1% of 2.0
    S_r = np.array([[4.0, 1.0, 10.0], [2.0, -1.0, 5.0]])  # value part | normaliser column
    o_g = o_r.copy(); o_g[1, 0] = 0.51; o_g[1, 1] = 0.011   # |d| 0.01 (rel 0.02) and 0.01 (excluded)
    S_g = S_r.copy(); S_g[0, 1] = 1.004                      # |d| 0.004, rel 0.004; normwise 0.004/4
    p = b.parity_vs_oracle([o_g], [S_g], [(o_r, S_r)], dv, 1e-4)
    assert p["heads"] == 1
    assert abs(p["normwise"]["out"] - 0.01 / 2.0) < 1e-12
    assert abs(p["elementwise_ge_1pct"]["out"] - 0.02) < 1e-12
    assert abs(p["normwise"]["state"] - 0.001) < 1e-12
    assert abs(p["elementwise_ge_1pct"]["state"] - 0.004) < 1e-12
    assert p["normwise"]["normaliser"] == 0.0 and p["elementwise_ge_1pct"]["normaliser"] == 0.0
    # all elements, |r| floored at 1e-6 max|r|: the small output 0.001 (error 0.01) dominates
    assert abs(p["elementwise_floor_1e-6"]["out"] - float(f"{0.01 / (0.001 + 2e-6):.3g}")) < 1e-9
    assert abs(p["elementwise_floor_1e-6"]["state"] - float(f"{0.004 / (1.0 + 4e-6):.3g}")) < 1e-12
    assert p["ok"] is False
    exact = b.parity_vs_oracle([o_r], [S_r], [(o_r, S_r)], dv, 1e-4)
    assert exact["ok"] and max(exact["normwise"].values()) == 0.0
