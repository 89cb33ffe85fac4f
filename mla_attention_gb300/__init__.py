"""libmla: the Multi-head Latent Attention forward on one GB300 (sm_103a).

The compute path is the CUDA library libmla.so (built in-tree by
mla_attention_gb300.build); this package is a thin ctypes binding over its C
ABI (include/mla.h) plus the seeded input generators used by tests and the
bench.  Importing the package does not load the library; the first call does,
and fails loudly if it was not built.
"""
from ._lib import (MLAError, check_device_status, exported_symbols, inject_stall, lib, mla_decode,
                   mla_absorb_q, mla_decode_ex, mla_decode_fp8, mla_decode_noalloc, mla_merge_lse, mla_project_out, mla_rope_append,
                   mla_prefill, mla_prefill_split, mla_prefill_varlen, mla_sparse, set_tile_keys, set_spin_limit, workspace)

__all__ = ["MLAError", "check_device_status", "exported_symbols", "inject_stall", "lib", "mla_decode",
           "mla_absorb_q", "mla_decode_ex", "mla_decode_fp8", "mla_decode_noalloc", "mla_merge_lse", "mla_project_out", "mla_rope_append",
           "mla_prefill", "mla_prefill_split", "mla_prefill_varlen", "mla_sparse", "set_tile_keys", "set_spin_limit",
           "workspace"]
