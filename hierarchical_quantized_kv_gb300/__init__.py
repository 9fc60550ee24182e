"""GB300-native QuantSpec hierarchical quantized KV cache: decode attention
over C_U / C_L nibble planes plus the fp16 double buffer, quantize-on-flush,
and append / rollback bookkeeping, as a C-ABI CUDA library (``libqs.so``).

``hierarchical_quantized_kv_gb300.qs`` is the ctypes binding (import it
explicitly; importing this package loads nothing).
"""
