"""GB300 (sm_103a) W4A16 + paged-GQA single-token decode library.

The compute lives in ``libw4a16_gb300.so`` (hand-written CUDA kernels behind
the C ABI in ``include/w4a16.h``); ``api`` is its torch-tensor binding and
``synth`` the seeded synthetic-input generator.  Importing the package does
not load CUDA; the first API call does, and fails loudly if the library has
not been built.
"""
import importlib

__all__ = ["api", "synth", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
