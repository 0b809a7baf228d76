"""GB300-native (sm_103a) DeepSeek-V4 C128 sparse-attention KV compressor.

``compress_norm_rope_store`` runs the whole path on the GPU through the C-ABI library
``libc128compress.so`` (built from ``csrc/`` by ``build.build()``); the binding only marshals
arguments. Importing the package itself loads nothing; the library is loaded on first use.
"""
import importlib

__all__ = ["compress_norm_rope_store"]


def __getattr__(name):
    if name == "compress_norm_rope_store":
        return importlib.import_module(".binding", __name__).compress_norm_rope_store
    raise AttributeError(name)
