"""Simple Gated Linear Attention on NVIDIA GB300 (sm_103a).

The compute lives in the C-ABI library ``libgla.so`` (hand-written CUDA); this
package holds its thin Python binding (``gated_linear_rnn_gb300.gla``), the
build step and the seeded input generators.  Importing the package does not
load the library; ``gla`` loads it on first use and raises if it is missing.
"""
__all__ = ["gla", "inputs", "build"]
