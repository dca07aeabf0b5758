"""GB300-native Q8_0 Llama forward.

The compute path is the C-ABI CUDA library built from ``csrc/`` (header
``include/llama_q8.h``); ``binding`` is its ctypes wrapper and ``synth`` the
seeded synthetic-input generator. Import ``q8_quantized_llama_gb300.binding``
for the library; importing this package alone loads nothing.
"""
