"""B300-native forward pass of a top-k routed MoE SwiGLU FFN layer.

The compute path is the C-ABI library ``libmoe.so`` (hand-written sm_103a CUDA);
``sparse_conditional_moe_b300.moe`` is its thin ctypes binding.  Importing this
package does not load the library; the first call into the binding does, and
it raises if the library has not been built.
"""
__all__ = ["accounting"]
