"""GB300-native log-linear attention: chunked forward, Fenwick decode, Gated DeltaNet.

The compute lives in ``libllattn.so`` (CUDA for sm_103a behind a C ABI,
declared in ``include/ll_attn.h``).  ``binding`` marshals torch tensors into
that ABI; ``synth`` draws seeded synthetic inputs.  Importing the package does
not load the library; ``binding.lib()`` does, and raises if it is missing.
"""

__all__ = ["binding", "synth"]


def __getattr__(name):
    if name == "binding":
        from . import binding
        return binding
    if name == "synth":
        from . import synth
        return synth
    raise AttributeError(name)
