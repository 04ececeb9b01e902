"""GB300-native verify-side rejection sampler for speculative decoding.

The compute path is the C-ABI library ``libspecreject.so`` (hand-written sm_103a
CUDA kernels, declared in ``include/spec_reject.h``); ``binding`` marshals torch
tensors into it.  ``workloads`` draws the seeded synthetic inputs.
"""
