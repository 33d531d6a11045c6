"""GB300-native quantised GEMV + norm decode-step library.

``quantised_gemv_norm_gb300.dq`` is the thin ctypes binding over the C-ABI
library ``libdq.so`` (built from ``csrc/`` for sm_103a); ``synth`` draws seeded
synthetic inputs; ``ledger`` holds the byte and roofline arithmetic used to
report bandwidth.  Importing this package does not load the CUDA library.
"""
