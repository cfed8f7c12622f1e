"""TokenGate pruned-prefill hot path for NVIDIA B300 (sm_103a).

The compute runs in ``libtokengate.so`` (hand-written CUDA kernels behind a
C ABI, declared in ``include/tokengate.h``); ``tokengate`` is the thin Python
binding with the same entry-point names, and ``synth`` holds the seeded input
generators."""
