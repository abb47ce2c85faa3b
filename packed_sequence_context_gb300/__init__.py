"""GB300-native causal attention over packed THD tensors with an emulated
P2P (ring) context-parallel decomposition.

The compute path is the C-ABI library ``libthdattn.so`` (hand-written CUDA for
sm_103a); ``packed_sequence_context_gb300.thd_attn`` is its thin ctypes
binding.  Importing this package does not load the library; the binding
loads it on first use and raises if it is missing.
"""

__all__ = ["inputs", "thd_attn"]
