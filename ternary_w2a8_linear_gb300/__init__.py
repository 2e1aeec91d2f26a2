"""GB300-native W2A8 ternary linear (sm_103a).

The compute lives in the C-ABI library ``libbitmtp_linear.so`` (declared in
``include/bitmtp_linear.h``); ``ternary_w2a8_linear_gb300.linear`` is the thin
ctypes binding over it.  ``inputs`` holds the seeded synthetic workloads.
"""
