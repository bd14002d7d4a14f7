"""seg_la on GB300: Bailing-style segmented lightning attention behind a C ABI.

The computation runs in hand-written sm_103a CUDA kernels (csrc/), reached through the C ABI of
include/la.h; this package holds the ctypes binding (binding.py), the in-tree build (_build.py)
and the seeded synthetic workloads (workloads.py).
"""
from .binding import (LAError, commit_accepted, decode, decode_gqa, extend, extend_gqa,  # noqa
                      extend_gqa_workspace_size, extend_noalloc, extend_workspace_size, load,
                      poll_error, set_balanced, set_column_split, set_persistent, set_wait_limit, slopes,
                      verify_chain, verify_tree)
