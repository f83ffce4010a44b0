"""libattnfuse: RoPE + causal softmax attention forward on GB300 (sm_103a).

The CUDA library is loaded lazily on first use (see :mod:`attention_rope_causal_gb300.binding`), so
importing the package or its input generator needs no GPU.
"""
__all__ = ["inputs"]
