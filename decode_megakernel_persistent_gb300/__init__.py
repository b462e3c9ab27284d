"""Batch-1 Llama-style decode as one persistent CUDA megakernel on GB300 (sm_103a).

The compute path is the C-ABI library ``libll.so`` built from ``csrc/``;
``ll`` is its thin ctypes binding. Importing this package loads nothing: the
library is opened on first use and its absence raises.
"""
