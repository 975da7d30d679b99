"""Seeded synthetic inputs shared by the oracle tests, the CUDA-path tests and the bench.

This package draws random numbers and lays out input *structure* only: shapes,
sequence lengths, which physical block holds which logical block, which
sequences share a prefix.  It contains none of the attention arithmetic and none
of the cache address arithmetic; both the oracle and the CUDA library consume
what it returns.
"""
from .gen import *  # noqa: F401,F403
