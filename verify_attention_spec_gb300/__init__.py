"""GB300-native paged decode/verify attention and speculative rejection sampling.

The compute lives in ``libvas.so`` (hand-written sm_103a CUDA behind a C ABI declared in
``include/vas.h``).  ``verify_attention_spec_gb300.binding`` marshals arguments to it and
raises if the library has not been built; there is no CPU fallback.
``verify_attention_spec_gb300.workloads`` only generates seeded synthetic inputs and
``verify_attention_spec_gb300._build`` compiles the library.
"""
import importlib

_SUBMODULES = ("binding", "workloads", "_build")
__all__ = ["binding", "workloads"]


def __getattr__(name):
    if name in _SUBMODULES:
        return importlib.import_module(f".{name}", __name__)
    if name.startswith("_"):
        raise AttributeError(name)
    return getattr(importlib.import_module(".binding", __name__), name)
