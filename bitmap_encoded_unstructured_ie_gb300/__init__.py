"""GB300-native bitmap-encoded unstructured-sparse SpMM / spMspV.

The compute runs in the CUDA library ``libus.so`` (C ABI declared in
``include/us.h``); :mod:`.binding` marshals arguments to it through ctypes.
Importing the package does not load the library; the first call does, and it
raises if the library has not been built.
"""
__all__ = ["binding", "workloads"]
