"""GB300-native PISA pyramid Top-K block selector.

The compute path lives in the C-ABI library built from ``csrc/`` (see
``include/pisa.h``); :mod:`pyramid_top_block_mean_gb300.pisa` is its thin
ctypes binding.  Importing the binding loads the library and raises if it is
missing: there is no CPU fallback.
"""
__all__ = ["pisa", "workloads"]
