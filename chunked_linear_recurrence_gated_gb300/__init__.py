"""GB300-native chunk-level Gated DeltaNet state transition (forward and backward).

The compute path is a C-ABI shared library of hand-written sm_103a CUDA kernels
(``csrc/``); ``gdn`` is its thin ctypes binding. Importing the package does not
load the library; the first call into ``gdn`` does, and fails loudly if it has
not been built.
"""
