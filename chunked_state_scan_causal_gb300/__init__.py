"""Chunked causal linear attention for GB300 (sm_103a): Python binding of liblinattn.

The binding is argument marshalling only; every step runs in the CUDA library.
"""
