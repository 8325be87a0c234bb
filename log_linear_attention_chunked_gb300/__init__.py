"""GB300-native log-linear attention: chunked forward, Fenwick decode, Gated DeltaNet.

The compute lives in ``libllattn.so`` (CUDA for sm_103a behind a C ABI,
declared in ``include/ll_attn.h``).  ``binding`` marshals torch tensors into
that ABI; ``synth`` draws seeded synthetic inputs.  Importing the package does
not load the library; ``binding.lib()`` does, and raises if it is missing.
"""

import importlib

__all__ = ["binding", "synth", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
