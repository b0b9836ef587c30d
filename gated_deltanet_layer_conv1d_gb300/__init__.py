"""Gated DeltaNet token mixer (conv1d -> gated delta rule -> gated RMSNorm) for GB300.

The compute lives in ``libgdn.so`` (hand-written CUDA for sm_103a behind a C ABI,
declared in ``include/gdn.h``).  ``gated_deltanet_layer_conv1d_gb300.gdn`` is the thin
ctypes binding over it; ``workloads`` holds the seeded synthetic inputs.
Importing this package does not load the CUDA library.
"""
