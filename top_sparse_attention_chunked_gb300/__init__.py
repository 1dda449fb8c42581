"""libdsa: dynamic sparse attention (indexer -> radix top-k -> sparse GQA
attention) on one GB300, as hand-written CUDA for sm_103a behind a C ABI
(include/dsa.h). This package holds the CUDA sources, the in-tree build and
the ctypes binding; importing it does not load the library."""
from . import dsa  # noqa: F401
from .dsa import (DsaError, DsaProblem, alloc_workspace, dsa_index_scores,  # noqa: F401
                  dsa_read_device_status, dsa_sparse_attn_decode, dsa_sparse_attn_prefill,
                  dsa_timing_read, dsa_timing_select, dsa_topk, dsa_version,
                  dsa_workspace_size, load_library, make_problem, problem_for)
