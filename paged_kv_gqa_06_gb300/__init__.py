"""Paged-KV decode attention for GB300 (sm_103a).

The operations, implemented as hand-written CUDA kernels behind a C ABI
(``include/forge_paged.h``, ``libforge_paged.so``):

  * ``forge_paged_kv_append`` -- scatter each sequence's new K/V token into
    its slot of the paged block pool;
  * ``forge_paged_gqa_decode`` -- grouped-query attention of one new query
    token per sequence over that sequence's cached K/V, read through its
    block table; long contexts are cut into splits whose partial results
    the last split to finish merges, in the same launch;
  * ``forge_paged_prefill`` -- causal attention of a run of new query tokens
    per sequence (a prompt, or the next chunk of one) over the paged cache;
  * ``forge_kv_pool_*`` / ``forge_batch_*`` (``include/forge_serving.h``) --
    the KV block pool and the continuous-batching step driver that produce
    the block tables, context lengths and slot mapping those calls read.

The Python functions of the same names (``paged_kv_gqa_06_gb300.binding``)
only marshal torch tensors into the C descriptors.  The CUDA library is
loaded on first use; if it is missing the call raises -- there is no CPU
fallback.
"""
from __future__ import annotations

__all__ = [
    "forge_paged_kv_append",
    "forge_paged_gqa_decode",
    "forge_paged_append_gqa_decode",
    "forge_paged_qk_append_gqa_decode",
    "forge_rope_cos_sin_table",
    "forge_paged_gqa_decode_ex",
    "forge_paged_gqa_decode_noalloc",
    "forge_paged_prefill",
    "forge_paged_gqa_decode_workspace_bytes",
    "forge_paged_gqa_decode_plan",
    "forge_paged_get_device_error",
    "forge_kv_pool_create",
    "forge_kv_pool_destroy",
    "forge_kv_pool_add",
    "forge_kv_pool_grow",
    "forge_kv_pool_release",
    "forge_kv_pool_free_blocks",
    "forge_kv_pool_used_blocks",
    "forge_kv_pool_sequence",
    "forge_batch_create",
    "forge_batch_destroy",
    "forge_batch_submit",
    "forge_batch_step",
    "forge_batch_rows",
    "forge_batch_events",
    "forge_batch_apply",
]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
