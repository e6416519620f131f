"""Quantized-KV MLA attention for GB300: KV8 / TQ4 / K2V4 codecs and decode/prefill kernels."""
