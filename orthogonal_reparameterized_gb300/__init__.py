"""POET-X layer on one NVIDIA GB300: a C-ABI CUDA library (``libpoetx.so``, sm_103a) and its
thin Python binding.

``poetx`` is the binding (import it explicitly; it loads the library on first use and
fails loudly if it is missing).  ``inputs`` is the seeded synthetic input generator.
"""
