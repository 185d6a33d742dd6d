"""Paged K/V attention for GB300 (sm_103a): a C-ABI CUDA library
(``include/pkv.h``, sources in ``csrc/``) with a thin ctypes binding."""
from . import workloads  # noqa: F401  (seeded input generators)
from .pkv import (  # noqa: F401
    kv_scatter_slots, paged_attention, paged_attention_workspace_size, merge_attn_states,
    rotate_rows, rope_write_kv_paged, copy_kv_slots, paged_attention_no_alloc, lib, PkvError)
