"""GB300-native prefill MoE expert layer: GPU routing + 4-bit grouped GEMM.

The public calls live in :mod:`routing_q4_grouped_gb300.moeq4` (a thin ctypes
binding over the C-ABI library ``libmoeq4.so``). Importing this package does
not load the library; ``synth`` (seeded inputs) stays importable on machines
without a GPU.
"""

__all__ = ["moeq4", "synth"]


def __getattr__(name):
    if name in __all__:
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
