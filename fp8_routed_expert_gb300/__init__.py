"""GB300-native routed Mixture-of-Experts FFN layer with blockwise-FP8 experts.

The compute path is the C-ABI library ``libfp8moe.so`` (hand-written sm_103a
kernels); this package is its thin Python binding.
"""
from ._lib import C, MoEError, exported_functions, lib  # noqa: F401
from .layer import ExpertCache, MoELayer  # noqa: F401
