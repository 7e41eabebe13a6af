"""GB300-native differential-attention head forward (sm_103a).

The compute path is the C-ABI library ``libdiffattn.so`` built from ``csrc/``;
``ops`` is its thin ctypes binding.  Importing this package does not load the
library; the first call into ``ops`` does, and raises if it is missing.
"""
__all__ = ["ops", "workloads"]
