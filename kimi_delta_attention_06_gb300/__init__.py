"""GB300-native Kimi Delta Attention (KDA) hot path: chunked prefill and decode.

The compute lives in a C-ABI CUDA library (``libkda.so``, built for sm_103a
from ``csrc/``); ``kimi_delta_attention_06_gb300.kda`` is a thin ctypes
binding with the same entry-point names.  Importing this package does not
load the library; the first call does, and fails loudly when it is missing.
"""
