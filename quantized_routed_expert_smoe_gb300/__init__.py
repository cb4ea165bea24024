"""libsmoe: the prompt-chunk routed-expert block of a mixture-of-experts layer on GB300 (sm_103a).

The compute lives in the CUDA library libsmoe.so (C ABI: include/smoe.h); ``binding`` is its thin Python binding
with the same call names, and ``synth`` makes the seeded synthetic inputs.  Importing the package does not load the
library; the first call does, and raises when it is missing.
"""
import importlib

from . import synth  # noqa: F401

__all__ = ["synth", "binding"]


def __getattr__(name):
    if name == "binding":
        return importlib.import_module(__name__ + ".binding")
    raise AttributeError(name)
