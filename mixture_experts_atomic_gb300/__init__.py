"""GB300-native dropless top-K MoE layer (MoEBlaze): index-only dispatch,
gather-fused tcgen05 expert GEMMs and fused combine, behind a C ABI.

The compute path lives in ``libmoeblaze.so`` (built from ``csrc/``); the
Python side (``binding``) only marshals pointers, sizes and streams.
"""
__all__ = ["binding", "inputs", "layer"]
