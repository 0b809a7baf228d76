"""CPU oracle for the DeepSeek-V4 C128 KV compressor (compress -> RMSNorm -> FP8/UE8M0 + RoPE
-> paged k_cache store).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's CPU-baseline
leg are the only code allowed to import this package. The CUDA library never calls it and
shares no code with it; the two meet only in the seeded inputs of
``deepseek_v4_sparse_c128_gb300.inputs``.

The arithmetic lives in ``c128_oracle.c`` (plain C, binary64 softmax, exact variance); this
module builds it with the host C compiler and wraps it with ctypes. Each C function cites the
passage of the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "c128_oracle.c")
_LIB = os.path.join(_HERE, "libc128oracle.so")
_lock = threading.Lock()
_lib = None

HEAD = 512
TOKEN_STRIDE = 576
SCALE_DIM = 8
# token / scale bytes per k_cache slot of each cache format (0: sparse attention, 1: indexer FP8,
# 2: indexer MXFP4)
FORMAT_BYTES = {0: (576, 8), 1: (128, 4), 2: (64, 4)}


class Cfg(ctypes.Structure):
    _fields_ = [("head", ctypes.c_int32), ("rope", ctypes.c_int32), ("ratio", ctypes.c_int32),
                ("overlap", ctypes.c_int32), ("state_width", ctypes.c_int32), ("format", ctypes.c_int32)]


def build(force: bool = False) -> str:
    """Compile the oracle (``cc -O2 -ffp-contract=off``) unless an up-to-date build exists."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cc = os.environ.get("CC", "cc")
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call([cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                           "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i64, i32p, i64p = ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
            f32p, u8p = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_uint8)
            L.c128o_bf16.argtypes = [ctypes.c_float]
            L.c128o_bf16.restype = ctypes.c_uint16
            L.c128o_e4m3.argtypes = [ctypes.c_float]
            L.c128o_e4m3.restype = ctypes.c_uint8
            L.c128o_rsqrt.argtypes = [ctypes.c_float]
            L.c128o_rsqrt.restype = ctypes.c_float
            L.c128o_ceil_log2.argtypes = [ctypes.c_float]
            L.c128o_ceil_log2.restype = ctypes.c_int
            L.c128o_mean_square_512.argtypes = [f32p]
            L.c128o_mean_square_512.restype = ctypes.c_float
            L.c128o_epilogue.argtypes = [f32p, f32p, ctypes.c_float, f32p, u8p, u8p]
            L.c128o_epilogue.restype = None
            L.c128o_compress_window.argtypes = [ctypes.POINTER(f32p), f32p]
            L.c128o_compress_window.restype = None
            L.c128o_forward.argtypes = [i64, i32p, i64p, i64p, i32p, i64, i64, i64, f32p, i64, i64, i64,
                                        f32p, ctypes.c_float, f32p, i64, i64, u8p, i64, i64, i64, i64p,
                                        f32p, i64p, i64]
            L.c128o_forward.restype = ctypes.c_int
            L.c128o_e2m1.argtypes = [ctypes.c_float]
            L.c128o_e2m1.restype = ctypes.c_uint8
            L.c128o_mean_square_128.argtypes = [f32p]
            L.c128o_mean_square_128.restype = ctypes.c_float
            for name in ("c128o_epilogue_indexer_fp8", "c128o_epilogue_indexer_mxfp4"):
                getattr(L, name).argtypes = [f32p, f32p, ctypes.c_float, f32p, u8p, u8p]
                getattr(L, name).restype = None
            L.c128o_forward_ex.argtypes = [ctypes.POINTER(Cfg), i64, i32p, i64p, i64p, i32p, i64, i64, i64, f32p,
                                           i64, i64, i64, i64, f32p, ctypes.c_float, f32p, i64, i64, u8p, i64, i64,
                                           i64, i64p, f32p, i64p, i64]
            L.c128o_forward_ex.restype = ctypes.c_int
            L.c128o_bf16_n.argtypes = [f32p, ctypes.POINTER(ctypes.c_uint16), i64]
            L.c128o_bf16_n.restype = None
            L.c128o_e4m3_n.argtypes = [f32p, u8p, i64]
            L.c128o_e4m3_n.restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return np.ascontiguousarray(a)


# ------------------------------------------------------------------------------- scalar pieces
def bf16_bits(x: float) -> int:
    return int(lib().c128o_bf16(ctypes.c_float(x)))


def e4m3_code(x: float) -> int:
    return int(lib().c128o_e4m3(ctypes.c_float(x)))


def ceil_log2(x: float) -> int:
    return int(lib().c128o_ceil_log2(ctypes.c_float(x)))


def rsqrt(x: float) -> np.float32:
    return np.float32(lib().c128o_rsqrt(ctypes.c_float(x)))


def bf16_bits_array(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.zeros(x.shape, np.uint16)
    lib().c128o_bf16_n(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint16), x.size)
    return out


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.zeros(x.shape, np.uint8)
    lib().c128o_e4m3_n(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint8), x.size)
    return out


def e2m1_code(x: float) -> int:
    return int(lib().c128o_e2m1(ctypes.c_float(x)))


def mean_square_128(c: np.ndarray) -> np.float32:
    c = _c(c, np.float32)
    assert c.shape == (128,)
    return np.float32(lib().c128o_mean_square_128(_ptr(c, ctypes.c_float)))


def epilogue_indexer(fmt: int, comp32: np.ndarray, rms_w: np.ndarray, eps: float, cos_sin_row: np.ndarray):
    """Indexer epilogue of one 128-wide compressed vector: fmt 1 -> (128 e4m3 bytes, 4 bytes of
    fp32 scale), fmt 2 -> (64 bytes of E2M1 pairs, 4 UE8M0 bytes)."""
    comp32, rms_w, cs = _c(comp32, np.float32), _c(rms_w, np.float32), _c(cos_sin_row, np.float32)
    nt, ns = FORMAT_BYTES[fmt]
    tok, sc = np.zeros(nt, np.uint8), np.zeros(ns, np.uint8)
    fn = lib().c128o_epilogue_indexer_fp8 if fmt == 1 else lib().c128o_epilogue_indexer_mxfp4
    fn(_ptr(comp32, ctypes.c_float), _ptr(rms_w, ctypes.c_float), ctypes.c_float(eps), _ptr(cs, ctypes.c_float),
       _ptr(tok, ctypes.c_uint8), _ptr(sc, ctypes.c_uint8))
    return tok, sc


def mean_square_512(c: np.ndarray) -> np.float32:
    c = _c(c, np.float32)
    assert c.shape == (HEAD,)
    return np.float32(lib().c128o_mean_square_512(_ptr(c, ctypes.c_float)))


def epilogue(comp32: np.ndarray, rms_w: np.ndarray, eps: float, cos_sin_row: np.ndarray):
    """RMSNorm + quant + RoPE of one compressed vector -> (576 token bytes, 8 scale bytes)."""
    comp32 = _c(comp32, np.float32)
    rms_w = _c(rms_w, np.float32)
    cs = _c(cos_sin_row, np.float32)
    tok = np.zeros(TOKEN_STRIDE, np.uint8)
    sc = np.zeros(SCALE_DIM, np.uint8)
    lib().c128o_epilogue(_ptr(comp32, ctypes.c_float), _ptr(rms_w, ctypes.c_float), ctypes.c_float(eps),
                         _ptr(cs, ctypes.c_float), _ptr(tok, ctypes.c_uint8), _ptr(sc, ctypes.c_uint8))
    return tok, sc


def compress_rows(rows: np.ndarray) -> np.ndarray:
    """Softmax-weighted sum over a window given as a [128, 1024] array of state rows."""
    rows = _c(rows, np.float32)
    assert rows.shape == (128, 1024)
    ptrs = (ctypes.POINTER(ctypes.c_float) * 128)(
        *[ctypes.cast(rows.ctypes.data + i * 4096, ctypes.POINTER(ctypes.c_float)) for i in range(128)])
    out = np.zeros(HEAD, np.float32)
    lib().c128o_compress_window(ptrs, _ptr(out, ctypes.c_float))
    return out


# ------------------------------------------------------------------------------------ whole op
def forward(problem, k_cache: Optional[np.ndarray] = None, tokens: Optional[Sequence[int]] = None,
            comp_out: Optional[np.ndarray] = None, threads: int = 1) -> int:
    """Run the op on ``problem`` (a ``deepseek_v4_sparse_c128_gb300.inputs.Problem`` with a numpy
    state) writing into ``k_cache`` (default: a copy of ``problem.k_cache``; pass an array to
    update in place). ``tokens`` restricts the work to those token indices. Returns the error bits.
    """
    L = lib()
    state = problem.state
    assert isinstance(state, np.ndarray) and state.dtype == np.float32 and state.flags.c_contiguous
    ttr = _c(problem.token_to_req, np.int32)
    pos = _c(problem.positions, np.int64)
    slot = _c(problem.slot_mapping, np.int64)
    bt = _c(problem.block_table, np.int32)
    kvs = _c(problem.kv_slot_mapping, np.int64)
    rms_w = _c(problem.rms_w, np.float32)
    cs = _c(problem.cos_sin, np.float32)
    if k_cache is None:
        k_cache = problem.k_cache.copy()
    assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous
    T = pos.shape[0]
    if comp_out is not None:
        assert comp_out.dtype == np.float32 and comp_out.shape == (T, HEAD) and comp_out.flags.c_contiguous
    all_tok = np.arange(T, dtype=np.int64) if tokens is None else np.asarray(tokens, dtype=np.int64)
    chunks = np.array_split(all_tok, max(1, threads)) if threads > 1 else [all_tok]

    def run(sub: np.ndarray) -> int:
        sub = np.ascontiguousarray(sub, dtype=np.int64)
        return L.c128o_forward(
            T, _ptr(ttr, ctypes.c_int32), _ptr(pos, ctypes.c_int64), _ptr(slot, ctypes.c_int64),
            _ptr(bt, ctypes.c_int32), bt.shape[0], bt.shape[1], bt.shape[1],
            _ptr(state, ctypes.c_float), state.shape[0], 8 * 1024, 1024,
            _ptr(rms_w, ctypes.c_float), ctypes.c_float(problem.eps),
            _ptr(cs, ctypes.c_float), cs.shape[0], cs.shape[1],
            _ptr(k_cache, ctypes.c_uint8), k_cache.shape[0], problem.kv_block_size,
            k_cache.shape[1] * k_cache.shape[2], _ptr(kvs, ctypes.c_int64),
            _ptr(comp_out, ctypes.c_float) if comp_out is not None else None,
            _ptr(sub, ctypes.c_int64), sub.shape[0])

    if len(chunks) == 1:
        err = run(chunks[0])
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:  # ctypes drops the GIL during each call
            err = 0
            for e in ex.map(run, chunks):
                err |= e
    return err


def problem_cfg(problem) -> Cfg:
    return Cfg(getattr(problem, "head", 512), 64, getattr(problem, "ratio", 128), getattr(problem, "overlap", 0),
               getattr(problem, "state_width", 512), getattr(problem, "fmt", 0))


def forward_ex(problem, k_cache: Optional[np.ndarray] = None, tokens: Optional[Sequence[int]] = None,
               comp_out: Optional[np.ndarray] = None, threads: int = 1) -> int:
    """The op for any configuration (head, compress ratio, overlap, state width, cache format) the
    problem carries; same conventions as forward(). comp_out is [T, head]."""
    L = lib()
    cfg = problem_cfg(problem)
    state = problem.state
    assert isinstance(state, np.ndarray) and state.dtype == np.float32 and state.flags.c_contiguous
    ttr, pos = _c(problem.token_to_req, np.int32), _c(problem.positions, np.int64)
    slot, bt = _c(problem.slot_mapping, np.int64), _c(problem.block_table, np.int32)
    kvs, rms_w = _c(problem.kv_slot_mapping, np.int64), _c(problem.rms_w, np.float32)
    cs = _c(problem.cos_sin, np.float32)
    if k_cache is None:
        k_cache = problem.k_cache.copy()
    assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous
    T = pos.shape[0]
    if comp_out is not None:
        assert comp_out.dtype == np.float32 and comp_out.shape == (T, cfg.head) and comp_out.flags.c_contiguous
    all_tok = np.arange(T, dtype=np.int64) if tokens is None else np.asarray(tokens, dtype=np.int64)
    chunks = np.array_split(all_tok, max(1, threads)) if threads > 1 else [all_tok]
    NB, BS, RW = state.shape

    def run(sub):
        sub = np.ascontiguousarray(sub, dtype=np.int64)
        return L.c128o_forward_ex(
            ctypes.byref(cfg), T, _ptr(ttr, ctypes.c_int32), _ptr(pos, ctypes.c_int64), _ptr(slot, ctypes.c_int64),
            _ptr(bt, ctypes.c_int32), bt.shape[0], bt.shape[1], bt.shape[1], _ptr(state, ctypes.c_float), NB, BS,
            BS * RW, RW, _ptr(rms_w, ctypes.c_float), ctypes.c_float(problem.eps), _ptr(cs, ctypes.c_float),
            cs.shape[0], cs.shape[1], _ptr(k_cache, ctypes.c_uint8), k_cache.shape[0], problem.kv_block_size,
            k_cache.shape[1] * k_cache.shape[2], _ptr(kvs, ctypes.c_int64),
            _ptr(comp_out, ctypes.c_float) if comp_out is not None else None, _ptr(sub, ctypes.c_int64), sub.shape[0])

    if len(chunks) == 1:
        err = run(chunks[0])
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            err = 0
            for e in ex.map(run, chunks):
                err |= e
    assert err >= 0, "unsupported configuration"
    return err


def forward_k_cache(problem, **kw) -> np.ndarray:
    """Convenience: the k_cache after the op (starting from ``problem.k_cache``)."""
    kc = problem.k_cache.copy()
    forward(problem, k_cache=kc, **kw)
    return kc
