"""GB300-native routed Mixture-of-Experts FFN forward.

The compute path lives in ``libmoe.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/moe.h``); :mod:`mixture_experts_ffn_gb300.moe` is
the thin ctypes binding over it.  The binding is imported lazily so that the
input generator (:mod:`.synth`) can be used without the library.
"""
import importlib

__all__ = ["moe", "synth"]


def __getattr__(name):
    if name in ("moe", "synth", "build"):
        return importlib.import_module(f".{name}", __name__)
    mod = importlib.import_module(".moe", __name__)
    try:
        return getattr(mod, name)
    except AttributeError:
        raise AttributeError(name) from None
