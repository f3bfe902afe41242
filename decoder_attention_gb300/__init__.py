"""GB300 (sm_103a) attention step of a rotary, grouped-query decoder layer.

The C-ABI library libdecattn.so (include/decattn.h) does all the work; ``_abi`` binds it with ctypes and
``step`` strings its four entry points together for one layer. Submodules load lazily, so that the
synthetic-input module can be imported on a machine where the library has not been built.
"""
import importlib

__all__ = ["_abi", "step", "inputs", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
