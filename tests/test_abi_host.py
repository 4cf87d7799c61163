"""CPU checks of the C ABI: the library loads, exports every symbol the header
declares, and its host-only logic (sizes, feature ordering, work planning,
argument validation) is right. No kernel is launched here."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from fixed_state_recurrence_phi_b300 import build as tsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def T():
    tsa_build.build()
    from fixed_state_recurrence_phi_b300 import tsa
    return tsa


def _header_functions():
    src = open(os.path.join(ROOT, "include", "tsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tsa_[a-z_]+)\s*\(", src)))


def test_exports_match_header(T):
    declared = _header_functions()
    assert declared == sorted(T.EXPORTS)
    lib = ctypes.CDLL(T.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    # the ELF dynamic symbol table agrees
    out = os.popen(f"nm -D --defined-only {T.LIB_PATH}").read()
    for name in declared:
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_sizes(T):
    for d in (1, 2, 16, 32):
        for n in range(1, 5):
            assert T.feature_dim(d, n) == sum(math.comb(d + m - 1, m) for m in range(n))
    assert T.feature_dim(0, 3) == 0 and T.feature_dim(16, 0) == 0
    cfg = T.Config(1, 1, 16, 64, 3)
    assert T.state_elems(cfg) == 9945 == (1 + 16 + 136) * 65
    assert T.state_pad_dim(16, 3) == 156
    assert T.state_bytes(T.Config(64, 16, 16, 64, 3)) == 64 * 16 * 156 * 65 * 4
    assert T.feature_dim(16, 4) == 969 and T.feature_dim(32, 3) == 561


@pytest.mark.parametrize("d,n", [(16, 1), (16, 2), (16, 3), (16, 4), (16, 5), (32, 3)])
def test_feature_order_matches_oracle(T, d, n):
    """The CUDA feature table (rows of the state) enumerates the same monomials
    in the same order with the same 1/sqrt(a!) weights as the oracle."""
    from oracle import tsa_oracle as O
    idx, w = T.feature_index(d, n)
    want = [t for m in range(n) for t in O.monomials(d, m)]
    got = [tuple(int(i) for i in row if i >= 0) for row in idx]
    assert got == want
    ww = np.array([1.0 / math.sqrt(O._alpha_factorial(t)) for t in want], dtype=np.float32)
    assert np.array_equal(w, ww)


def test_order_five_plans(T):
    """n = 5 at d_k = 16 (4,845 features): the CUDA-core path, one value slice
    of d_v columns, both dtypes, from one span to many."""
    assert T.feature_dim(16, 5) == 4845 == 1 + 16 + 136 + 816 + 3876
    for dt in ("f32", "bf16"):
        for dv in (32, 64):
            for N in (1, 64, 300, 8192):
                p = T.prefill_plan(T.Config(1, 8, 16, dv, 5, dt), N, num_sms=148)
                assert p["path"] == T.TSA_PATH_SIMT and p["n_slices"] == 1 and p["slice_width"] == dv
                assert p["n_spans"] * p["chunks_per_span"] >= -(-N // 64)
    assert T.prefill_plan(T.Config(1, 8, 16, 64, 5), 8192, num_sms=148)["n_spans"] > 1


def test_plan_covers_all_chunks(T):
    for (B, H, N, d, dv, n) in [(1, 8, 8192, 16, 64, 3), (1, 1, 256, 16, 64, 3),
                                (64, 16, 65536, 16, 64, 3), (4, 16, 32768, 16, 64, 4),
                                (2, 32, 65536, 32, 128, 3), (1, 1, 1, 16, 64, 3),
                                (3, 5, 1000, 32, 32, 2)]:
        p = T.prefill_plan(T.Config(B, H, d, dv, n), N, num_sms=148)
        chunks = -(-N // p["chunk"])
        assert p["n_spans"] >= 1 and p["chunks_per_span"] >= 1
        assert p["n_spans"] * p["chunks_per_span"] >= chunks
        assert (p["n_spans"] - 1) * p["chunks_per_span"] < chunks   # no empty span
        assert p["n_slices"] * p["slice_width"] == dv
        assert p["smem_bytes"] <= 227 * 1024
        if p["n_spans"] > 1:
            assert p["launches"] == 3
            assert p["scratch_bytes"] == B * H * p["n_spans"] * T.state_pad_dim(d, n) * (dv + 1) * 4
        else:
            assert p["launches"] == 1 and p["scratch_bytes"] == 0
    # the 8-head, 8192-token prefill spreads each head over many spans
    assert T.prefill_plan(T.Config(1, 8, 16, 64, 3), 8192, num_sms=148)["n_spans"] >= 8


def test_plan_short_segments(T):
    """Short segments go to the shared-memory-resident path where the state
    fits; chunk = 16 asks for it at any length; chunk = 128 keeps the chunked
    tensor-core path."""
    for dt in ("f32", "bf16"):
        # bf16 segments of 17..64 tokens take the tensor-core append form instead
        n_max = 16 if dt == "bf16" else 32
        for N in (1, 16, 32):
            p = T.prefill_plan(T.Config(64, 16, 16, 64, 3, dt), N, num_sms=148)
            if N > n_max:
                assert p["path"] == T.TSA_PATH_TC and p["ctas_per_sm"] == 3, (dt, N, p)
                continue
            assert p["path"] == T.TSA_PATH_SHORT and p["chunk"] == 16, (dt, N, p)
            assert p["chunks_per_span"] == -(-N // 16) and p["launches"] == 1 and p["scratch_bytes"] == 0
            assert p["ctas_per_sm"] >= 2
        assert T.prefill_plan(T.Config(64, 16, 16, 64, 3, dt), 33, num_sms=148)["path"] != T.TSA_PATH_SHORT
        assert T.prefill_plan(T.Config(1, 1, 16, 64, 3, dt, chunk=16), 5000,
                              num_sms=148)["path"] == T.TSA_PATH_SHORT
        assert T.prefill_plan(T.Config(64, 16, 16, 64, 3, dt, chunk=128), 8,
                              num_sms=148)["path"] != T.TSA_PATH_SHORT
    # bf16 states the append form does not take keep the short path up to 32 tokens
    assert T.prefill_plan(T.Config(4, 4, 32, 128, 2, "bf16"), 32, num_sms=148)["path"] == T.TSA_PATH_SHORT
    # shared memory of the layout: state, phi(q) and phi(k) of a block, the
    # block's values and inputs, intra-block kernel values, the 8 warps'
    # readout partials and normaliser partials, feature codes and weights, and
    # the mbarrier, in fp32 words
    def words(d, dv, n):
        dpad = -(-T.feature_dim(d, n) // 4) * 4
        x = -(-(16 * (d + 1)) // 4) * 4
        return dpad * (dv + 1) + 2 * dpad * 16 + 16 * dv + 2 * x + 256 + 8 * 16 * dv + 8 * 16 + 2 * dpad + 4
    for (d, dv, n) in [(16, 64, 3), (16, 32, 3), (16, 128, 2), (32, 128, 2), (32, 32, 1)]:
        p = T.prefill_plan(T.Config(4, 4, d, dv, n, "f32", chunk=16), 40, num_sms=148)
        assert p["path"] == T.TSA_PATH_SHORT and p["smem_bytes"] == 4 * words(d, dv, n), (d, dv, n, p)
        assert p["smem_bytes"] <= 113 * 1024
    # states too large for shared memory keep the chunked paths
    for (d, dv, n) in [(16, 64, 4), (32, 64, 3), (16, 128, 3)]:
        assert T.prefill_plan(T.Config(4, 4, d, dv, n, "bf16"), 8, num_sms=148)["path"] != T.TSA_PATH_SHORT
        with pytest.raises(T.TsaError):
            T.prefill_plan(T.Config(4, 4, d, dv, n, "bf16", chunk=16), 8, num_sms=148)


def test_validation_codes(T):
    """Invalid arguments are rejected on the host before any CUDA call."""
    ok = T.Config(1, 1, 16, 64, 3)
    fake = 1 << 40   # aligned, never dereferenced: validation fails first
    cases = [
        (T.Config(1, 1, 8, 64, 3), T.TSA_ERR_UNSUPPORTED),
        (T.Config(1, 1, 16, 48, 3), T.TSA_ERR_UNSUPPORTED),
        (T.Config(1, 1, 16, 64, 6), T.TSA_ERR_UNSUPPORTED),
        (T.Config(1, 1, 16, 128, 5), T.TSA_ERR_UNSUPPORTED),  # order 4: one value slice only
        (T.Config(1, 1, 32, 64, 4), T.TSA_ERR_UNSUPPORTED),   # D = 6545 > 1024
        (T.Config(0, 1, 16, 64, 3), T.TSA_ERR_INVALID),
        (T.Config(1, 1, 16, 64, 0), T.TSA_ERR_INVALID),
    ]
    for cfg, code in cases:
        with pytest.raises(T.TsaError) as e:
            T.prefill(cfg, 10, fake, fake, fake, fake, fake, stream=0)
        assert e.value.status == code, cfg
        with pytest.raises(T.TsaError) as e:
            T.decode_step(cfg, fake, fake, fake, fake, fake, stream=0)
        assert e.value.status == code
    with pytest.raises(T.TsaError) as e:          # N < 0
        T.prefill(ok, -1, fake, fake, fake, fake, fake, stream=0)
    assert e.value.status == T.TSA_ERR_INVALID
    with pytest.raises(T.TsaError) as e:          # NULL states
        T.prefill(ok, 10, fake, fake, fake, fake, 0, stream=0)
    assert e.value.status == T.TSA_ERR_INVALID
    with pytest.raises(T.TsaError) as e:          # misaligned q
        T.prefill(ok, 10, fake + 4, fake, fake, fake, fake, stream=0)
    assert e.value.status == T.TSA_ERR_INVALID
    with pytest.raises(T.TsaError) as e:          # unknown flag bits
        T._check("tsa_prefill", T._lib.tsa_prefill(ctypes.byref(ok.c()), 10, fake, fake, fake, fake,
                                                   fake, 2, 0))
    assert e.value.status == T.TSA_ERR_INVALID
    with pytest.raises(T.TsaError) as e:          # NULL decode input
        T.decode_step(ok, 0, fake, fake, fake, fake, stream=0)
    assert e.value.status == T.TSA_ERR_INVALID
    nb = T.state_bytes(ok)
    with pytest.raises(T.TsaError) as e:          # partially overlapping merge
        T.state_merge(ok, fake, fake + 16 * (nb // 32), stream=0)
    assert e.value.status == T.TSA_ERR_INVALID
    assert "overlap" in T.last_error()
    with pytest.raises(T.TsaError) as e:
        T.prefill_plan(ok, -5, num_sms=148)
    assert e.value.status == T.TSA_ERR_INVALID
    # token coordinates are 32-bit: 2^31 - 1 tokens plan, 2^31 do not
    assert T.prefill_plan(ok, (1 << 31) - 1, num_sms=148)["n_spans"] >= 1
    with pytest.raises(T.TsaError) as e:
        T.prefill_plan(ok, 1 << 31, num_sms=148)
    assert e.value.status == T.TSA_ERR_INVALID and "2^31" in T.last_error()
    assert T.status_string(T.TSA_ERR_TIMEOUT) == "TSA_ERR_TIMEOUT"


def test_debug_hooks_validate(T):
    """The testing hooks take only their documented values (host only)."""
    for bad in (4, -1):
        with pytest.raises(T.TsaError) as e:
            T.debug_withhold_publication(bad)
        assert e.value.status == T.TSA_ERR_INVALID
    for good in (1, 2, 3, 0):
        T.debug_withhold_publication(good)
    T.debug_set_wait_limit(0)


def test_chunk_lengths_built(T):
    """fp32 prefill chunk lengths: 64 (CUDA cores), 128 (tensor cores) and
    16 (short segments); 256 is not built (refused on the host)."""
    for chunk, path in [(64, T.TSA_PATH_SIMT), (128, T.TSA_PATH_TC_F32), (16, T.TSA_PATH_SHORT)]:
        p = T.prefill_plan(T.Config(1, 8, 16, 64, 3, "f32", chunk), 8192, num_sms=148)
        assert p["chunk"] == chunk and p["path"] == path, (chunk, p)
    with pytest.raises(T.TsaError) as e:
        T.prefill_plan(T.Config(1, 8, 16, 64, 3, "f32", 256), 8192, num_sms=148)
    assert e.value.status == T.TSA_ERR_UNSUPPORTED


def test_release_and_debug_builds(T):
    """The release library has no device checks (tsa_debug_build() == 0, the
    self-test is refused before any launch); the debug build exports the same
    symbols and reports itself as the debug build (host only)."""
    assert T.LIB_PATH.endswith("libtsa.so") or os.environ.get("TSA_DEBUG") == "1"
    if not T.debug_build():
        assert T._lib.tsa_debug_check_selftest(None) == T.TSA_ERR_UNSUPPORTED
        assert "debug build" in T.last_error()
    assert T.status_string(T.TSA_ERR_DEVICE_CHECK) == "TSA_ERR_DEVICE_CHECK"
    dbg_path = tsa_build.build(debug=True)
    lib = ctypes.CDLL(dbg_path)
    lib.tsa_debug_build.restype = ctypes.c_int
    assert lib.tsa_debug_build() == 1
    out = os.popen(f"nm -D --defined-only {dbg_path}").read()
    for name in _header_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name
