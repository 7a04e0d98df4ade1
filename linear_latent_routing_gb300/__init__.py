"""GB300-native Gaussian Mixture Attention (GMA) forward pass.

The compute lives in ``libgma.so`` (hand-written sm_103a CUDA behind a C ABI, declared in
``include/gma.h``); ``linear_latent_routing_gb300.gma`` is the thin ctypes binding over it.
The binding is imported on demand so that host-only code (input generation) works without a
built library; it raises if the library is missing.
"""
__all__ = ["gma", "inputs"]
