"""Quantized KV cache for GB300: quantize-on-append and decode attention over
packed low-bit blocks, as a C-ABI CUDA library (libkvq.so) with a thin
Python binding (``bit_kv_cache_04_gb300.kvq``)."""
