"""GB300-native MoE FFN layer: 8-bit router, top-k, 4-bit group-64 SwiGLU
experts, shared expert and weighted combine, as hand-written CUDA for sm_103a
behind a small C ABI (``include/moe.h``).

``moe`` is the Python binding of that ABI (argument marshalling only);
``synth`` draws seeded synthetic layers and hidden states.
"""
