"""Split backward (B / W) of one Zero-Bubble pipeline stage on GB300 (sm_103a).

The compute path is the C-ABI library ``libzb.so`` built from ``csrc/``;
``binding`` wraps it with ctypes under the same names.  Importing this package
does not load the library: ``binding.lib()`` does, and raises if it is missing.
"""
