"""Frame-wise Gated DeltaNet forward scan on B300 (sm_103a).

The compute path is the C-ABI library ``libgdn.so`` built from ``csrc/``;
``binding`` marshals arguments to it.  Importing this package does not load the
library; the first call through ``binding`` does, and raises if it is missing.
"""
