"""ISD verify-and-propose on one B300: Python binding of libisd (the headers
under include/).

The computation runs in libisd.so (hand-written sm_103a CUDA); this package
marshals torch CUDA tensors into its C ABI.  ``workloads`` makes seeded
synthetic inputs.
"""
from .api import (ProposeOut, VerifyOut, isd_alpha, isd_kv_commit, isd_propose,  # noqa: F401
                  isd_propose_filtered, isd_propose_filtered_workspace_bytes, isd_propose_workspace_bytes,
                  isd_verify, isd_verify_filtered, isd_verify_filtered_workspace_bytes, isd_verify_propose,
                  isd_verify_propose_workspace_bytes, isd_verify_workspace_bytes, workspace)
