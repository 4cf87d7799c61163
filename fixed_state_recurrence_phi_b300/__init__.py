"""Truncated-Taylor fixed-state causal attention on NVIDIA B300 (sm_103a).

The compute path is libtsa.so (C ABI, include/tsa.h) built from csrc/; the
binding is `fixed_state_recurrence_phi_b300.tsa` (imported on first use, so that
the input generators and the build script load without the library).
"""
import importlib


def __getattr__(name):
    if name == "tsa":
        return importlib.import_module(__name__ + ".tsa")
    raise AttributeError(name)
