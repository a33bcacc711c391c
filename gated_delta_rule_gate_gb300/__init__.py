"""Gated delta rule recurrence on GB300 (sm_103a): a C-ABI CUDA library
(libgdn.so, declared in include/gdn.h) and a thin torch binding.

Entry points (same names as the C ABI):
    gdn_gate, gdn_recurrent_step, gdn_chunked_prefill,
    gdn_chunked_prefill_workspace_size, gdn_chunked_prefill_workspace_size_min,
    gdn_chunked_prefill_noalloc, gdn_status_string
"""
from ._native import GdnError, library_path, load  # noqa: F401
from .api import (gdn_chunked_prefill, gdn_chunked_prefill_noalloc,  # noqa: F401
                  gdn_chunked_prefill_workspace_size, gdn_chunked_prefill_workspace_size_min, gdn_gate,
                  gdn_recurrent_step,
                  gdn_status_string, make_problem)
