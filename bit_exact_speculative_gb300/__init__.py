"""Exact speculative verify for hybrid gated-delta-net / attention decoders on GB300.

The compute lives in ``libxv.so`` (CUDA for sm_103a, C ABI in ``include/xv.h``);
``bit_exact_speculative_gb300.xv`` is its thin Python binding and
``bit_exact_speculative_gb300.build`` compiles it in-tree.
"""
from . import xv  # noqa: F401

__all__ = ["xv"]
