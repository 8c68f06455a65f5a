"""GB300-native (sm_103a) kernels for position-independent caching of
linear-attention state: segment build of (T_C, S(C|0)), composition of cached
pairs in any order, and seam-window advance.

The compute path is ``libhypic.so`` (hand-written CUDA behind a C ABI, see
``include/hypic.h``); ``linear_attn_state_gb300.hypic`` is its thin Python
binding.  ``synth`` draws the seeded synthetic inputs.
"""
