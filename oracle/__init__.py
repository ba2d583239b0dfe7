"""Test-infrastructure oracle (float64, CPU) for paged MLA decode with DCP shards.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product library never imports it, and it never imports the
product library.
"""
from .mla_ref import (  # noqa: F401
    PAD_SLOT_ID,
    ref_abs_weighted,
    ref_attention_global,
    ref_build_pool,
    ref_cp_local_slot,
    ref_gather_pages,
    ref_local_len,
    ref_lse_merge,
    ref_mla_decode,
    ref_mla_decode_global,
    ref_owned_positions,
    ref_row_global_prefix,
    ref_scatter_kv,
)
