"""GB300-native paged decode/verify attention and speculative rejection sampling.

The compute lives in ``libvas.so`` (hand-written sm_103a CUDA behind a C ABI declared in
``include/vas.h``).  ``verify_attention_spec_gb300.binding`` marshals arguments to it and
raises if the library has not been built; there is no CPU fallback.
``verify_attention_spec_gb300.workloads`` only generates seeded synthetic inputs.
"""
import importlib

__all__ = ["binding", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f".{name}", __name__)
    binding = importlib.import_module(".binding", __name__)
    if hasattr(binding, name):
        return getattr(binding, name)
    raise AttributeError(name)
