"""GB300-native (sm_103a) DDTree verification round: build, tree attention, tree GDN,
walk and commit as hand-written CUDA kernels behind the C ABI of include/ddt.h.

``ddt`` is the thin binding (import it explicitly); ``synth`` holds the seeded input
generators.  Importing the package loads nothing.
"""
__all__ = ["ddt", "synth", "build_ext"]
