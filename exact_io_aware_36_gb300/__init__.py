"""Exact IO-aware attention (forward and backward) for one GB300 (sm_103a).

The compute path is the C-ABI library ``libfa`` (hand-written CUDA kernels);
``exact_io_aware_36_gb300.fa`` is its thin Python binding.  Importing the
package does not load the library; the binding loads it on first use and
raises if it is missing.
"""
__all__ = ["inputs", "fa"]
