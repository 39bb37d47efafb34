"""GB300-native (sm_103a) Mesa layer forward pass: chunked CG prefill and recurrent decode.

The compute runs in hand-written CUDA kernels behind a C ABI (``include/mesa.h``); the
``binding`` module marshals torch tensors into that ABI.  ``synth`` holds the seeded
input generators of the benchmark workloads.
"""
