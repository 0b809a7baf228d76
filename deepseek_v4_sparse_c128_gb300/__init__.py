"""GB300-native (sm_103a) DeepSeek-V4 C128 sparse-attention KV compressor.

``compress_norm_rope_store`` runs the whole path on the GPU through the C-ABI library
``libc128compress.so`` (built from ``csrc/``); the binding only marshals arguments.
"""
__all__ = ["compress_norm_rope_store"]


def __getattr__(name):
    if name in ("compress_norm_rope_store", "binding"):
        from . import binding
        return binding if name == "binding" else binding.compress_norm_rope_store
    raise AttributeError(name)
