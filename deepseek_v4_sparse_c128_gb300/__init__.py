"""GB300-native (sm_103a) DeepSeek-V4 C128 sparse-attention KV compressor.

``compress_norm_rope_store`` runs the whole path on the GPU through the C-ABI library
``libc128compress.so`` (built from ``csrc/`` by ``build.build()``); the binding only marshals
arguments. Importing the package itself loads nothing; the library is loaded on first use.

Use (torch tensors on the current device, the current stream)::

    from deepseek_v4_sparse_c128_gb300 import build, binding
    build.build()                       # once: compiles the library in-tree for sm_103a
    binding.compress_norm_rope_store(token_to_req_indices, positions, slot_mapping, block_table,
                                     state_cache, rms_w, eps, cos_sin_cache, k_cache,
                                     kv_slot_mapping, kv_block_size)
    # the other configurations of the fused kernels (C4 overlap, indexer FP8 / MXFP4 caches)
    cfg = binding.config(head_dim=128, compress_ratio=4, overlap=1, cache_format=binding.FORMAT_INDEXER_MXFP4)
    binding.compress_norm_rope_store_ex(cfg, token_to_req_indices, positions, slot_mapping, block_table,
                                        state_cache, rms_w, eps, cos_sin_cache, k_cache,
                                        kv_slot_mapping, kv_block_size)
    bits = binding.device_errors()      # out-of-range indices (tokens skipped), wait time-outs

Calls are asynchronous and CUDA-graph capturable after ``binding.reserve_workspace(max_tokens)``;
``binding.PreparedCall`` builds the descriptors once for repeated calls on the same tensors.
"""
import importlib

__all__ = ["compress_norm_rope_store", "compress_norm_rope_store_ex"]


def __getattr__(name):
    if name in __all__:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
