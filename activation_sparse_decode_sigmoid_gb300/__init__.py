"""GB300 (sm_103a) library for the PowerInfer decode hot path: a low-rank
activation predictor followed by a neuron-aware sparse FFN.

The compute lives in ``libpi.so`` (hand-written CUDA, C ABI declared in
``include/pi.h``).  ``activation_sparse_decode_sigmoid_gb300.pi`` is the thin
ctypes binding with the same entry-point names; ``workload`` draws the seeded
synthetic layers.  Nothing here falls back to a CPU path: if the extension is
missing, loading the binding raises.
"""
import importlib

__all__ = ["pi", "workload"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
