"""GB300-native (sm_103a) fused 2-D convolution layer and its companion ops.

The compute lives in ``lib/libacnn.so`` (CUDA kernels behind the C ABI of
``include/acnn.h``); ``acnn`` is its Python binding, ``network`` builds and
replays the layer graphs of the workloads, ``inputs`` draws seeded synthetic
inputs.  Importing the package does not load the library.
"""
__all__ = ["acnn", "inputs", "network", "build"]
