"""GB300-native hot path of batch speculative decoding: verify + realign behind a C-ABI library.

``specdec`` is the ctypes binding of ``libspecdec.so`` (imported on first use, and it raises if the
library has not been built); ``synth`` holds the seeded input generators; ``engine`` holds the
caller-side round state (ping-pong caches) used by the benchmark.
"""
__version__ = "0.1.0"


def __getattr__(name):
    if name in ("specdec", "engine", "synth"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
