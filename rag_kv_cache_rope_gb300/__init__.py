"""GB300-native selective KV-recompute ("blended") prefill for RAG.

The compute path is the C-ABI library ``libblend.so`` built from ``csrc/``; the
Python binding (``binding``) only marshals arguments.  Importing this package does
not load the library; ``binding.lib()`` does, and fails loudly if it is missing.
"""
