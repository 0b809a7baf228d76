"""ctypes binding of libc128compress (include/c128compress.h).

Argument marshalling only: torch tensors (or raw device pointers) become ``c128_tensor_t``
descriptors and the current torch CUDA stream becomes the call's stream. Every step of the op
runs in the library's CUDA kernels; there is no fallback path, and importing this module fails
loudly if the library cannot be loaded.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

C128_I32, C128_I64, C128_F32, C128_U8 = 1, 2, 3, 4
STATUS = {
    0: "C128_OK", 1: "C128_ERR_NULL_PTR", 2: "C128_ERR_DTYPE", 3: "C128_ERR_SHAPE", 4: "C128_ERR_STRIDE",
    5: "C128_ERR_ALIGN", 6: "C128_ERR_UNSUPPORTED", 7: "C128_ERR_ARG", 8: "C128_ERR_CUDA", 9: "C128_ERR_NOMEM",
    10: "C128_ERR_TOO_MANY_TOKENS", 11: "C128_ERR_CAPTURE",
}
NOALLOC_MAX_TOKENS = 65536  # C128_NOALLOC_MAX_TOKENS
DEV_BITS = {1: "BAD_REQ", 2: "BAD_BT_COL", 4: "BAD_BLOCK", 8: "BAD_COS_ROW", 16: "BAD_KV_SLOT", 32: "TIMEOUT"}

# Every entry point the header declares, with its ctypes signature.
EXPORTS = (
    "compress_norm_rope_store",
    "c128_compress_norm_rope_store_debug",
    "c128_compress_norm_rope_store_noalloc",
    "compress_norm_rope_store_ex",
    "c128_debug_stall_first_window",
    "c128_debug_stall_first_window_ex",
    "c128_status_string",
    "c128_reserve_workspace",
    "c128_release_stream",
    "c128_device_errors",
    "c128_kernel_timer_begin",
    "c128_kernel_timer_end",
    "c128_get_info",
    "c128_read_probe",
    "c128_release_all",
)


class Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


FORMAT_SPARSE_FP8, FORMAT_INDEXER_FP8, FORMAT_INDEXER_MXFP4 = 0, 1, 2


class Config(ctypes.Structure):
    """c128_config_t: head_dim, rope_head_dim, compress_ratio, overlap, state_width, cache_format."""
    _fields_ = [("head_dim", ctypes.c_int32), ("rope_head_dim", ctypes.c_int32), ("compress_ratio", ctypes.c_int32),
                ("overlap", ctypes.c_int32), ("state_width", ctypes.c_int32), ("cache_format", ctypes.c_int32)]


def config(head_dim=512, compress_ratio=128, overlap=0, state_width=None, cache_format=0, rope_head_dim=64) -> Config:
    sw = state_width if state_width is not None else head_dim * (1 + overlap)
    return Config(head_dim, rope_head_dim, compress_ratio, overlap, sw, cache_format)


class Info(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int32), ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("plan_tokens_per_cta", ctypes.c_int32), ("wait_timeout_ms", ctypes.c_int32),
                ("version", ctypes.c_int32)]


class C128Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({lib().c128_status_string(status).decode()})")


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (built in-tree by ``deepseek_v4_sparse_c128_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libc128compress.so not found at {path}; run deepseek_v4_sparse_c128_gb300.build.build()")
    L = ctypes.CDLL(path)
    T = ctypes.POINTER(Tensor)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    L.compress_norm_rope_store.argtypes = [T, T, T, T, T, T, ctypes.c_float, T, T, T, i64, vp]
    L.c128_compress_norm_rope_store_debug.argtypes = [T, T, T, T, T, T, ctypes.c_float, T, T, T, i64, T, vp]
    L.c128_compress_norm_rope_store_noalloc.argtypes = [T, T, T, T, T, T, ctypes.c_float, T, T, T, i64, vp]
    L.c128_debug_stall_first_window.argtypes = [T, T, T, T, T, T, ctypes.c_float, T, T, T, i64, vp]
    L.c128_debug_stall_first_window_ex.argtypes = [ctypes.POINTER(Config), T, T, T, T, T, T, ctypes.c_float, T, T,
                                                   T, i64, vp]
    L.compress_norm_rope_store_ex.argtypes = [ctypes.POINTER(Config), T, T, T, T, T, T, ctypes.c_float, T, T, T, i64,
                                              T, vp]
    L.c128_status_string.argtypes = [ctypes.c_int]
    L.c128_status_string.restype = ctypes.c_char_p
    L.c128_reserve_workspace.argtypes = [i64, vp]
    L.c128_release_stream.argtypes = [vp]
    L.c128_device_errors.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
    L.c128_kernel_timer_begin.argtypes = [vp]
    L.c128_kernel_timer_end.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
    L.c128_get_info.argtypes = [ctypes.POINTER(Info)]
    i32 = ctypes.c_int32
    L.c128_read_probe.argtypes = [vp, i64, i32, i32, i32, vp, vp]
    L.c128_release_all.argtypes = []
    for name in EXPORTS:
        if name != "c128_status_string":
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def lib() -> ctypes.CDLL:
    return load()


# ----------------------------------------------------------------------------- marshalling
_TORCH_DTYPES = None


def _dtype_code(t) -> int:
    global _TORCH_DTYPES
    import torch
    if _TORCH_DTYPES is None:
        _TORCH_DTYPES = {torch.int32: C128_I32, torch.int64: C128_I64, torch.float32: C128_F32,
                         torch.uint8: C128_U8}
    if t.dtype not in _TORCH_DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _TORCH_DTYPES[t.dtype]


def describe(t) -> Tensor:
    """c128_tensor_t of a torch tensor (any device; the library expects device memory)."""
    d = Tensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _dtype_code(t)
    d.ndim = t.dim()
    if d.ndim > 4:
        raise ValueError("at most 4 dimensions")
    for i in range(d.ndim):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, where: str):
    if rc != 0:
        raise C128Error(rc, where)


def compress_norm_rope_store(token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w,
                             eps: float, cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size: int,
                             stream=None, comp_out=None) -> None:
    """Run the C128 compressor on CUDA tensors (see include/c128compress.h for the contract).
    ``k_cache`` is updated in place. ``comp_out`` ([T, 512] fp32), if given, receives the fp32
    compressed vectors of the stored tokens (the debug entry point)."""
    L = lib()
    args = [describe(x) for x in (token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w)]
    cs, kc, kvs = describe(cos_sin_cache), describe(k_cache), describe(kv_slot_mapping)
    h = _stream_handle(stream)
    refs = [ctypes.byref(a) for a in args]
    if comp_out is None:
        rc = L.compress_norm_rope_store(*refs, ctypes.c_float(eps), ctypes.byref(cs), ctypes.byref(kc),
                                        ctypes.byref(kvs), int(kv_block_size), h)
        _check(rc, "compress_norm_rope_store")
    else:
        co = describe(comp_out)
        rc = L.c128_compress_norm_rope_store_debug(*refs, ctypes.c_float(eps), ctypes.byref(cs), ctypes.byref(kc),
                                                   ctypes.byref(kvs), int(kv_block_size), ctypes.byref(co), h)
        _check(rc, "c128_compress_norm_rope_store_debug")


def compress_norm_rope_store_ex(cfg: Config, token_to_req_indices, positions, slot_mapping, block_table, state_cache,
                                rms_w, eps: float, cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size: int,
                                stream=None, comp_out=None) -> None:
    """The op for any configuration of the pages' fused kernels (see include/c128compress.h):
    C4-style overlap, head-128 indexer caches in FP8 or MXFP4. ``comp_out`` ([T, head]) optional."""
    L = lib()
    descs = [describe(x) for x in (token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w)]
    cs, kc, kvs = describe(cos_sin_cache), describe(k_cache), describe(kv_slot_mapping)
    co = describe(comp_out) if comp_out is not None else None
    rc = L.compress_norm_rope_store_ex(ctypes.byref(cfg), *[ctypes.byref(a) for a in descs], ctypes.c_float(eps),
                                       ctypes.byref(cs), ctypes.byref(kc), ctypes.byref(kvs), int(kv_block_size),
                                       ctypes.byref(co) if co is not None else None, _stream_handle(stream))
    _check(rc, "compress_norm_rope_store_ex")


def debug_stall_first_window(token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w,
                             eps: float, cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size: int,
                             stream=None) -> None:
    """Test of the bounded waits (tests only): the C128 call with CTA 0's first stage never
    filled, so the kernel gives up after its wait limit and reports C128_DEV_TIMEOUT (read it with
    device_errors) instead of hanging. Needs more tokens than the GPU has SMs."""
    L = lib()
    descs = [describe(x) for x in (token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w)]
    cs, kc, kvs = describe(cos_sin_cache), describe(k_cache), describe(kv_slot_mapping)
    rc = L.c128_debug_stall_first_window(*[ctypes.byref(a) for a in descs], ctypes.c_float(eps), ctypes.byref(cs),
                                         ctypes.byref(kc), ctypes.byref(kvs), int(kv_block_size),
                                         _stream_handle(stream))
    _check(rc, "c128_debug_stall_first_window")


def debug_stall_first_window_ex(cfg, token_to_req_indices, positions, slot_mapping, block_table, state_cache,
                                rms_w, eps: float, cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size: int,
                                stream=None) -> None:
    """The same test of the bounded waits for compress_norm_rope_store_ex (tests only): CTA 0 of
    the small-window or indexer kernel leaves its first stage unfilled."""
    L = lib()
    descs = [describe(x) for x in (token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w)]
    cs, kc, kvs = describe(cos_sin_cache), describe(k_cache), describe(kv_slot_mapping)
    rc = L.c128_debug_stall_first_window_ex(ctypes.byref(cfg), *[ctypes.byref(a) for a in descs], ctypes.c_float(eps),
                                            ctypes.byref(cs), ctypes.byref(kc), ctypes.byref(kvs), int(kv_block_size),
                                            _stream_handle(stream))
    _check(rc, "c128_debug_stall_first_window_ex")


def compress_norm_rope_store_noalloc(token_to_req_indices, positions, slot_mapping, block_table, state_cache,
                                     rms_w, eps: float, cos_sin_cache, k_cache, kv_slot_mapping,
                                     kv_block_size: int, stream=None) -> None:
    """The entry point that allocates no device memory (its scratch is a static device array of
    NOALLOC_MAX_TOKENS tokens); same arguments and results as compress_norm_rope_store. For
    callers that must not allocate once running. Calls that overlap on the GPU race."""
    L = lib()
    descs = [describe(x) for x in (token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w)]
    cs, kc, kvs = describe(cos_sin_cache), describe(k_cache), describe(kv_slot_mapping)
    rc = L.c128_compress_norm_rope_store_noalloc(*[ctypes.byref(a) for a in descs], ctypes.c_float(eps),
                                                 ctypes.byref(cs), ctypes.byref(kc), ctypes.byref(kvs),
                                                 int(kv_block_size), _stream_handle(stream))
    _check(rc, "c128_compress_norm_rope_store_noalloc")


class PreparedCall:
    """compress_norm_rope_store with its descriptors built once, for repeated calls on the same
    tensors (serving loops, benchmarks): calling the object is a single C-ABI call. The tensors
    must stay alive and keep their storage; the stream is fixed when the object is built
    (default: the current torch stream). ``noalloc=True`` targets
    c128_compress_norm_rope_store_noalloc instead; ``comp_out`` targets the debug entry point."""

    def __init__(self, token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w, eps: float,
                 cos_sin_cache, k_cache, kv_slot_mapping, kv_block_size: int, stream=None, comp_out=None,
                 noalloc: bool = False, cfg: Optional[Config] = None):
        L = lib()
        self._keep = (token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w, cos_sin_cache,
                      k_cache, kv_slot_mapping, comp_out)
        d = [describe(x) for x in (token_to_req_indices, positions, slot_mapping, block_table, state_cache, rms_w)]
        cs, kc, kvs = describe(cos_sin_cache), describe(k_cache), describe(kv_slot_mapping)
        self._descs = (*d, cs, kc, kvs)
        args = [ctypes.byref(a) for a in d] + [ctypes.c_float(eps), ctypes.byref(cs), ctypes.byref(kc),
                                               ctypes.byref(kvs), ctypes.c_int64(int(kv_block_size))]
        if cfg is not None:
            self._cfg = cfg
            self._co = describe(comp_out) if comp_out is not None else None
            args = [ctypes.byref(self._cfg)] + args + [ctypes.byref(self._co) if self._co is not None else None]
            self._fn, self._name = L.compress_norm_rope_store_ex, "compress_norm_rope_store_ex"
        elif comp_out is not None:
            self._co = describe(comp_out)
            args.append(ctypes.byref(self._co))
            self._fn, self._name = L.c128_compress_norm_rope_store_debug, "c128_compress_norm_rope_store_debug"
        elif noalloc:
            self._fn, self._name = L.c128_compress_norm_rope_store_noalloc, "c128_compress_norm_rope_store_noalloc"
        else:
            self._fn, self._name = L.compress_norm_rope_store, "compress_norm_rope_store"
        args.append(ctypes.c_void_p(_stream_handle(stream)))
        self._args = tuple(args)

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc != 0:
            raise C128Error(rc, self._name)


def call_status(*args, **kw) -> int:
    """Like compress_norm_rope_store but returns the status code instead of raising."""
    try:
        compress_norm_rope_store(*args, **kw)
        return 0
    except C128Error as e:
        return e.status


def reserve_workspace(max_tokens: int, stream=None) -> None:
    _check(lib().c128_reserve_workspace(int(max_tokens), _stream_handle(stream)), "c128_reserve_workspace")


def release_stream(stream=None) -> None:
    """Return the stream's workspace and timer events (stream-ordered; before destroying it)."""
    _check(lib().c128_release_stream(_stream_handle(stream)), "c128_release_stream")


def device_errors(stream=None, clear: bool = True) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib().c128_device_errors(_stream_handle(stream), ctypes.byref(bits), int(clear)), "c128_device_errors")
    return int(bits.value)


class KernelTimer:
    """Sum of compress-kernel times (CUDA events on the launching stream) between enter and exit."""

    def __init__(self, stream=None):
        self.stream = stream
        self.total_ms = 0.0
        self.launches = 0

    def __enter__(self):
        _check(lib().c128_kernel_timer_begin(_stream_handle(self.stream)), "c128_kernel_timer_begin")
        return self

    def __exit__(self, *exc):
        ms, n = ctypes.c_double(0), ctypes.c_int64(0)
        _check(lib().c128_kernel_timer_end(_stream_handle(self.stream), ctypes.byref(ms), ctypes.byref(n)),
               "c128_kernel_timer_end")
        self.total_ms, self.launches = ms.value, n.value
        return False


def info() -> dict:
    i = Info()
    _check(lib().c128_get_info(ctypes.byref(i)), "c128_get_info")
    return {f: getattr(i, f) for f, _ in Info._fields_}


def read_probe(buf, xor_out, threads_per_cta: int = 512, ctas_per_sm: int = 4, loads_in_flight: int = 8,
               stream=None) -> None:
    """Stream the whole contiguous device tensor ``buf`` once (c128_read_probe) and XOR its 32-bit
    words into the int32 device tensor ``xor_out`` (one element, zero it first)."""
    if not buf.is_contiguous():
        raise ValueError("read_probe needs a contiguous tensor")
    nbytes = buf.numel() * buf.element_size()
    _check(lib().c128_read_probe(buf.data_ptr(), nbytes, int(threads_per_cta), int(ctas_per_sm),
                                 int(loads_in_flight), xor_out.data_ptr(), _stream_handle(stream)),
           "c128_read_probe")


def release_all() -> None:
    _check(lib().c128_release_all(), "c128_release_all")
