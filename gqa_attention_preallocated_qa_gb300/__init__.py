"""GB300-native GQA attention hot path: fused QK-RMSNorm + RoPE + KV-cache
append, causal GQA prefill attention (tcgen05 / TMA) and split-KV decode
attention, behind the C ABI declared in ``include/qa.h``.

Importing the package loads nothing; ``binding`` loads the CUDA library and
fails loudly if it is missing.
"""
__version__ = "0.1.0"
