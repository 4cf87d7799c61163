"""Thin ctypes binding of libtsa.so (include/tsa.h), with the same names.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI. Tensors are passed as raw device pointers (torch is
used for device memory and streams). If the library is not built, importing
this module raises: there is no fallback path. With TSA_DEBUG=1 in the
environment the debug build (libtsa_debug.so: the same kernels with device-side
checks before each TMEM, shared-memory operand, TMA and state access) is
loaded instead.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtsa_debug.so" if os.environ.get("TSA_DEBUG") == "1" else "libtsa.so")

TSA_OK, TSA_ERR_INVALID, TSA_ERR_UNSUPPORTED, TSA_ERR_CUDA, TSA_ERR_TIMEOUT, TSA_ERR_DEVICE_CHECK = range(6)
TSA_F32, TSA_BF16 = 0, 1
TSA_PREFILL_ACCUMULATE = 1
TSA_PATH_SIMT, TSA_PATH_TC, TSA_PATH_TC_F32, TSA_PATH_SHORT = 0, 1, 2, 3

# Every symbol include/tsa.h declares (checked by the CPU test suite).
EXPORTS = (
    "tsa_feature_dim", "tsa_state_pad_dim", "tsa_state_elems", "tsa_state_bytes",
    "tsa_feature_index", "tsa_feature_map", "tsa_prefill_plan", "tsa_prefill", "tsa_prefill_noalloc", "tsa_prefill_states",
    "tsa_decode_step",
    "tsa_state_merge", "tsa_state_to_canonical", "tsa_sync_status",
    "tsa_status_string", "tsa_last_error",
    "tsa_debug_set_wait_limit", "tsa_debug_withhold_publication",
    "tsa_debug_build", "tsa_debug_check_selftest",
)


class TsaConfig(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("d_k", ctypes.c_int),
                ("d_v", ctypes.c_int), ("n_terms", ctypes.c_int), ("dtype", ctypes.c_int),
                ("chunk", ctypes.c_int)]


class TsaPlan(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_int), ("slice_width", ctypes.c_int), ("n_slices", ctypes.c_int),
                ("n_spans", ctypes.c_int), ("chunks_per_span", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("launches", ctypes.c_int),
                ("smem_bytes", ctypes.c_size_t), ("scratch_bytes", ctypes.c_size_t),
                ("path", ctypes.c_int), ("cluster", ctypes.c_int)]


class TsaError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {status_string(status)}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -m fixed_state_recurrence_phi_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, U, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint, ctypes.c_size_t
    C = ctypes.POINTER(TsaConfig)
    sig = {
        "tsa_feature_dim": (SZ, [I, I]),
        "tsa_state_pad_dim": (SZ, [I, I]),
        "tsa_state_elems": (SZ, [C]),
        "tsa_state_bytes": (SZ, [C]),
        "tsa_feature_index": (I, [I, I, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float)]),
        "tsa_feature_map": (I, [I, I, I64, P, P, P]),
        "tsa_prefill_plan": (I, [C, I64, I, ctypes.POINTER(TsaPlan)]),
        "tsa_prefill": (I, [C, I64, P, P, P, P, P, U, P]),
        "tsa_prefill_noalloc": (I, [C, I64, P, P, P, P, P, U, P]),
        "tsa_prefill_states": (I, [C, I64, P, P, P, U, P]),
        "tsa_decode_step": (I, [C, P, P, P, P, P, P]),
        "tsa_state_merge": (I, [C, P, P, P]),
        "tsa_state_to_canonical": (I, [C, P, P, P]),
        "tsa_sync_status": (I, [P]),
        "tsa_status_string": (ctypes.c_char_p, [I]),
        "tsa_last_error": (ctypes.c_char_p, []),
        "tsa_debug_set_wait_limit": (I, [ctypes.c_uint64]),
        "tsa_debug_withhold_publication": (I, [I]),
        "tsa_debug_build": (I, []),
        "tsa_debug_check_selftest": (I, [P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


_lib = _load()


def status_string(s: int) -> str:
    return _lib.tsa_status_string(int(s)).decode()


def last_error() -> str:
    return _lib.tsa_last_error().decode()


def _check(fn: str, s: int):
    if s != TSA_OK:
        raise TsaError(fn, s, last_error())


@dataclass(frozen=True)
class Config:
    B: int
    H: int
    d_k: int
    d_v: int
    n_terms: int
    dtype: str = "f32"   # "f32" | "bf16"
    chunk: int = 0

    def c(self) -> TsaConfig:
        return TsaConfig(self.B, self.H, self.d_k, self.d_v, self.n_terms,
                         {"f32": TSA_F32, "bf16": TSA_BF16}[self.dtype], self.chunk)


def _cfg(cfg) -> ctypes.POINTER(TsaConfig):
    c = cfg.c() if isinstance(cfg, Config) else cfg
    return ctypes.byref(c)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def feature_dim(d_k: int, n_terms: int) -> int:
    return _lib.tsa_feature_dim(d_k, n_terms)


def state_pad_dim(d_k: int, n_terms: int) -> int:
    return _lib.tsa_state_pad_dim(d_k, n_terms)


def state_elems(cfg) -> int:
    return _lib.tsa_state_elems(_cfg(cfg))


def state_bytes(cfg) -> int:
    return _lib.tsa_state_bytes(_cfg(cfg))


def feature_index(d_k: int, n_terms: int):
    """(idx [D, F], weight [D]) of the state rows, F = max(3, n_terms - 1)."""
    D = feature_dim(d_k, n_terms)
    F = max(3, n_terms - 1)
    idx = (ctypes.c_int * (F * max(D, 1)))()
    w = (ctypes.c_float * max(D, 1))()
    _check("tsa_feature_index", _lib.tsa_feature_index(d_k, n_terms, idx, w))
    return np.array(idx[:F * D], dtype=np.int32).reshape(D, F), np.array(w[:D], dtype=np.float32)


def feature_map(d_k: int, n_terms: int, x, out, stream=None):
    """phi(x) of the rows of x ([rows, d_k] fp32) into out ([rows, D] fp32)."""
    _check("tsa_feature_map", _lib.tsa_feature_map(int(d_k), int(n_terms), int(x.shape[0]), _ptr(x), _ptr(out),
                                                   _stream(stream)))


def prefill_plan(cfg, N: int, num_sms: int = 0) -> dict:
    p = TsaPlan()
    _check("tsa_prefill_plan", _lib.tsa_prefill_plan(_cfg(cfg), int(N), int(num_sms), ctypes.byref(p)))
    return {f: getattr(p, f) for f, _ in TsaPlan._fields_}


def prefill(cfg, N: int, q, k, v, out, states, accumulate: bool = False, stream=None):
    flags = TSA_PREFILL_ACCUMULATE if accumulate else 0
    _check("tsa_prefill", _lib.tsa_prefill(_cfg(cfg), int(N), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                           _ptr(states), flags, _stream(stream)))


def prefill_noalloc(cfg, N: int, q, k, v, out, states, accumulate: bool = False, stream=None):
    """tsa_prefill without any device allocation (fixed 16 MiB scratch array;
    see include/tsa.h for the limits)."""
    flags = TSA_PREFILL_ACCUMULATE if accumulate else 0
    _check("tsa_prefill_noalloc",
           _lib.tsa_prefill_noalloc(_cfg(cfg), int(N), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                    _ptr(states), flags, _stream(stream)))


def prefill_states(cfg, N: int, k, v, states, accumulate: bool = False, stream=None):
    """The state sum of N tokens (no outputs); see include/tsa.h."""
    flags = TSA_PREFILL_ACCUMULATE if accumulate else 0
    _check("tsa_prefill_states", _lib.tsa_prefill_states(_cfg(cfg), int(N), _ptr(k), _ptr(v), _ptr(states), flags,
                                                         _stream(stream)))


def decode_step(cfg, q, k, v, out, states, stream=None):
    _check("tsa_decode_step", _lib.tsa_decode_step(_cfg(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                                   _ptr(states), _stream(stream)))


def state_merge(cfg, a, b, stream=None):
    _check("tsa_state_merge", _lib.tsa_state_merge(_cfg(cfg), _ptr(a), _ptr(b), _stream(stream)))


def state_to_canonical(cfg, states, dst, stream=None):
    _check("tsa_state_to_canonical",
           _lib.tsa_state_to_canonical(_cfg(cfg), _ptr(states), _ptr(dst), _stream(stream)))


def sync_status(stream=None):
    _check("tsa_sync_status", _lib.tsa_sync_status(_stream(stream)))


def debug_set_wait_limit(ns: int):
    """Testing hook: the bound of every wait between warp roles (0 = default)."""
    _check("tsa_debug_set_wait_limit", _lib.tsa_debug_set_wait_limit(int(ns)))


def debug_withhold_publication(what: int):
    """Testing hook: 1 = the fp32 output pass withholds its first publication;
    2 = rank 0 of each CTA pair withholds its first exchange publication;
    3 = the bf16 append form withholds its output's completion."""
    _check("tsa_debug_withhold_publication", _lib.tsa_debug_withhold_publication(int(what)))


def debug_build() -> bool:
    """True when the loaded library is the debug build (device-side checks)."""
    return bool(_lib.tsa_debug_build())


def debug_check_selftest(stream=None):
    """Debug build: queue one kernel whose TMEM-column check fails on purpose
    (no TMEM access); the next sync_status raises TSA_ERR_DEVICE_CHECK."""
    _check("tsa_debug_check_selftest", _lib.tsa_debug_check_selftest(_stream(stream)))


# ---- small torch conveniences (allocation only) ----------------------------

def torch_dtype(cfg):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16}[cfg.dtype]


def new_states(cfg, device="cuda"):
    """Zeroed fp32 state buffer of tsa_state_bytes(cfg) bytes."""
    import torch
    return torch.zeros(state_bytes(cfg) // 4, dtype=torch.float32, device=device)


def canonical_states(cfg, states):
    """Device copy of `states` in the canonical layout [B, H, D, d_v + 1]."""
    import torch
    D = feature_dim(cfg.d_k, cfg.n_terms)
    dst = torch.empty((cfg.B, cfg.H, D, cfg.d_v + 1), dtype=torch.float32, device=states.device)
    state_to_canonical(cfg, states, dst)
    return dst
