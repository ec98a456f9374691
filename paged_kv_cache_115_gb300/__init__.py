"""GB300-native paged KV-cache decode path.

The compute lives in ``libpagedkv.so`` (hand-written sm_103a CUDA behind a C
ABI, declared in ``include/pagedkv.h``).  ``ops`` is the thin torch-facing
binding; ``blockmgr`` / ``workloads`` generate block tables and synthetic
inputs on the host; ``accounting`` counts bytes.  Importing this package does
not load the CUDA library; importing ``ops`` does, and fails loudly if it is
missing.
"""

__all__ = ["accounting", "blockmgr", "workloads"]
