"""Qwen3 attention core (QK-Norm -> RoPE -> causal GQA) for one GB300 (sm_103a).

The compute runs in the CUDA library ``libq3a.so`` behind the C ABI of
``include/q3a.h``; ``qwen3_qk_norm_gb300.binding`` is a thin ctypes layer over
it. Importing this package loads nothing: the library is loaded on the first
call and an ``ImportError`` is raised if it was not built.
"""
__all__ = ["binding", "inputs", "accounting"]
