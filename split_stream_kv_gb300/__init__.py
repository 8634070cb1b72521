"""GB300 (sm_103a) split-stream KV codec and packed-KV decode attention.

The compute lives in liblynx.so (C ABI, include/lynx.h); `lynx` is its
ctypes binding and `synth` draws seeded synthetic inputs.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "lynx"]


def __getattr__(name):
    if name == "lynx":
        import importlib
        return importlib.import_module(__name__ + ".lynx")
    raise AttributeError(name)
