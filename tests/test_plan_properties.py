"""Properties every prefill plan must have, over random shapes (host only, the
library's planner at 148 SMs): the spans cover every chunk with none empty,
the value slices tile d_v, a CTA pair only where the path is the bf16 tensor
cores, scratch exactly for the span states when there are several spans, the
occupancy within what one SM holds, and the one-slice global-state layout for
n = 5. Shapes the library does not build are refused with TSA_ERR_UNSUPPORTED,
never planned."""
import math

import pytest
from hypothesis import given, settings, strategies as st

from fixed_state_recurrence_phi_b300 import build as tsa_build

tsa_build.build()
from fixed_state_recurrence_phi_b300 import tsa as T  # noqa: E402

SMEM_PER_SM = 228 * 1024

shapes = st.tuples(
    st.integers(1, 8), st.integers(1, 64),          # B, H
    st.sampled_from([16, 32]), st.sampled_from([32, 64, 128]),   # d_k, d_v
    st.integers(1, 5), st.sampled_from(["f32", "bf16"]),          # n, dtype
    st.sampled_from([0, 0, 16, 64, 128]),           # chunk
    st.integers(1, 200_000))                         # N


@settings(max_examples=200, deadline=None)
@given(shapes)
def test_plan_properties(shape):
    B, H, d, dv, n, dtype, chunk, N = shape
    cfg = T.Config(B, H, d, dv, n, dtype, chunk)
    try:
        p = T.prefill_plan(cfg, N, num_sms=148)
    except T.TsaError as e:
        assert e.status == T.TSA_ERR_UNSUPPORTED, (shape, e)
        return
    chunks = -(-N // p["chunk"])
    assert p["chunk"] in (16, 64, 128)
    if chunk:
        assert p["chunk"] == chunk
    assert p["n_spans"] >= 1 and p["chunks_per_span"] >= 1
    assert p["n_spans"] * p["chunks_per_span"] >= chunks
    assert (p["n_spans"] - 1) * p["chunks_per_span"] < chunks            # no empty span
    assert p["n_slices"] * p["slice_width"] == dv
    assert p["cluster"] in (1, 2)
    if p["cluster"] == 2:
        assert p["path"] == T.TSA_PATH_TC and dtype == "bf16"
    assert 1 <= p["ctas_per_sm"] <= 3
    assert p["ctas_per_sm"] * p["smem_bytes"] <= SMEM_PER_SM
    state = T.state_bytes(T.Config(B, H, d, dv, n, dtype))
    if p["n_spans"] > 1:
        assert p["scratch_bytes"] == state * p["n_spans"] and p["launches"] == 3
    else:
        assert p["scratch_bytes"] == 0 and p["launches"] == 1
    if n == 5:
        assert d == 16 and dv in (32, 64) and p["path"] == T.TSA_PATH_SIMT and p["n_slices"] == 1
    D = sum(math.comb(d + m - 1, m) for m in range(n))
    assert D <= 1024 or (d, n) == (16, 5)
