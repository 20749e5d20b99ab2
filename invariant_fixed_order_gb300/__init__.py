"""Batch-invariant transformer forward step for one GB300 (sm_103a).

The compute path is the C-ABI library ``libbi.so`` built from ``csrc/``;
``invariant_fixed_order_gb300.bi`` is its thin ctypes binding.  Importing this
package does not load the library; importing ``.bi`` does, and fails loudly if
it has not been built.
"""
__all__ = ["config", "synth", "roofline"]
