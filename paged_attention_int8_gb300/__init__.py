"""paged_attention_int8_gb300: paged attention over a q8 KV cache on GB300.

The compute lives in a C-ABI CUDA library (``libpaq8.so``, built for sm_103a);
this package is its thin ctypes binding.  ``kv_store`` quantizes K/V rows to
the q8 format (int8 codes, one fp16 scale per token, kv head and 32 channels)
and scatters them into a block-paged cache; ``paged_attention`` runs unified
causal prefill + decode over that cache and returns bf16 output and fp32 LSE;
``merge_attn_states`` merges two such results over disjoint key sets by their
LSEs.

Importing the package does not load the CUDA library; the first call does, and
fails loudly if it has not been built.
"""
from __future__ import annotations

__all__ = ["kv_store", "kv_store_norm_rope", "kv_store_f8v4", "paged_attention",
           "paged_attention_f8v4", "paged_attention_noalloc", "merge_attn_states",
           "workspace_size", "check_status",
           "auto_num_splits", "Status", "PagedAttentionError", "library_path"]


def __getattr__(name):
    if name in __all__:
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
