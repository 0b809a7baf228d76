"""Host-only checks of the C-ABI library (no GPU needed): it builds for sm_103a, loads, exports
every function include/c128compress.h declares, and rejects bad arguments before touching CUDA.
Also checks that the CUDA path and the oracle share no code."""
import ctypes
import os
import re

import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "c128compress.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M))
                  - {"if", "while", "for", "return", "sizeof"})


def test_header_declarations_are_exported(L):
    names = declared_functions()
    assert "compress_norm_rope_store" in names
    assert sorted(binding.EXPORTS) == names
    for n in names:
        assert hasattr(L, n), n


def test_symbols_visible_to_nm():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in syms, n


def test_status_strings(L):
    for code in range(0, 11):
        s = L.c128_status_string(code)
        assert s and s != b"unknown status", code
    assert L.c128_status_string(99) == b"unknown status"


FAKE = 1 << 20  # an aligned address that validation never dereferences


def _t(shape, dtype, data=FAKE, strides=None):
    d = binding.Tensor()
    d.data = data
    d.dtype = dtype
    d.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for n in reversed(shape):
            strides.insert(0, acc)
            acc *= n
    for i, (n, s) in enumerate(zip(shape, strides)):
        d.shape[i], d.stride[i] = n, s
    return d


def _args(T=0, **over):
    I32, I64, F32, U8 = binding.C128_I32, binding.C128_I64, binding.C128_F32, binding.C128_U8
    a = dict(ttr=_t([T], I32), pos=_t([T], I64), slot=_t([T], I64), bt=_t([4, 64], I32),
             state=_t([64, 8, 1024], F32), rms=_t([512], F32), eps=1e-6, cs=_t([512, 64], F32),
             kc=_t([4, 2, 584], U8), kvs=_t([T], I64), bs=2)
    a.update(over)
    return a


def _call(L, a):
    r = lambda x: ctypes.byref(x) if x is not None else None
    return L.compress_norm_rope_store(r(a["ttr"]), r(a["pos"]), r(a["slot"]), r(a["bt"]), r(a["state"]),
                                      r(a["rms"]), ctypes.c_float(a["eps"]), r(a["cs"]), r(a["kc"]), r(a["kvs"]),
                                      a["bs"], None)


def test_empty_call_is_ok_without_gpu(L):
    assert _call(L, _args(T=0)) == 0


@pytest.mark.parametrize("case,code", [
    ("null_desc", 1), ("null_data", 1), ("pos_dtype", 2), ("state_dtype", 2), ("kc_dtype", 2),
    ("T_mismatch", 3), ("state_rank", 3), ("kc_width", 3), ("pos_stride", 4), ("state_inner_stride", 4),
    ("kc_inner", 4), ("state_misaligned", 5), ("state_stride_odd", 5), ("kc_stride0", 5),
    ("block8", 6), ("row1024", 6), ("head512", 6), ("rope64", 6), ("bs_mismatch", 7), ("bs_zero", 7),
])
def test_validation_codes(L, case, code):
    I32, I64, F32, U8 = binding.C128_I32, binding.C128_I64, binding.C128_F32, binding.C128_U8
    T = 5
    a = _args(T=T)
    if case == "null_desc":
        a["bt"] = None
    elif case == "null_data":
        a["slot"] = _t([T], I64, data=None)
    elif case == "pos_dtype":
        a["pos"] = _t([T], I32)
    elif case == "state_dtype":
        a["state"] = _t([64, 8, 1024], U8)
    elif case == "kc_dtype":
        a["kc"] = _t([4, 2, 584], I32)
    elif case == "T_mismatch":
        a["kvs"] = _t([T + 1], I64)
    elif case == "state_rank":
        a["state"] = _t([64, 8192], F32)
    elif case == "kc_width":
        a["kc"] = _t([4, 2, 583], U8)
    elif case == "pos_stride":
        a["pos"] = _t([T], I64, strides=[2])
    elif case == "state_inner_stride":
        a["state"] = _t([64, 8, 1024], F32, strides=[16384, 2048, 2])
    elif case == "kc_inner":
        a["kc"] = _t([4, 2, 584], U8, strides=[1168, 584, 2])
    elif case == "state_misaligned":
        a["state"] = _t([64, 8, 1024], F32, data=FAKE + 4)
    elif case == "state_stride_odd":
        a["state"] = _t([64, 8, 1024], F32, strides=[8 * 1026, 1026, 1])
    elif case == "kc_stride0":
        a["kc"] = _t([4, 1, 584], U8, strides=[588, 584, 1])
        a["bs"] = 1
    elif case == "block8":
        a["state"] = _t([64, 16, 1024], F32)
    elif case == "row1024":
        a["state"] = _t([64, 8, 2048], F32)
    elif case == "head512":
        a["rms"] = _t([128], F32)
    elif case == "rope64":
        a["cs"] = _t([512, 32], F32)
    elif case == "bs_mismatch":
        a["bs"] = 4
    elif case == "bs_zero":
        a["bs"] = 0
    assert _call(L, a) == code


def test_misaligned_comp_out_is_rejected(L):
    a = _args(T=5)
    r = ctypes.byref
    comp = _t([5, 512], binding.C128_F32, data=FAKE + 8)
    rc = L.c128_compress_norm_rope_store_debug(r(a["ttr"]), r(a["pos"]), r(a["slot"]), r(a["bt"]), r(a["state"]),
                                               r(a["rms"]), ctypes.c_float(1e-6), r(a["cs"]), r(a["kc"]),
                                               r(a["kvs"]), 2, r(comp), None)
    assert rc == 5


def test_debug_entry_requires_comp_out(L):
    a = _args(T=0)
    r = ctypes.byref
    rc = L.c128_compress_norm_rope_store_debug(r(a["ttr"]), r(a["pos"]), r(a["slot"]), r(a["bt"]), r(a["state"]),
                                               r(a["rms"]), ctypes.c_float(1e-6), r(a["cs"]), r(a["kc"]),
                                               r(a["kvs"]), 2, None, None)
    assert rc == 1
    comp = _t([0, 512], binding.C128_F32)
    rc = L.c128_compress_norm_rope_store_debug(r(a["ttr"]), r(a["pos"]), r(a["slot"]), r(a["bt"]), r(a["state"]),
                                               r(a["rms"]), ctypes.c_float(1e-6), r(a["cs"]), r(a["kc"]),
                                               r(a["kvs"]), 2, r(comp), None)
    assert rc == 0


def _sources(folder, exts):
    for dp, _, fs in os.walk(os.path.join(ROOT, folder)):
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(dp, f)


def test_oracle_and_cuda_path_share_no_code():
    pkg = "deepseek_v4_sparse_c128_gb300"
    for f in _sources(pkg, (".py", ".cu", ".h", ".cuh", ".cpp")):
        text = open(f).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
        assert "c128_oracle" not in text and "libc128oracle" not in text, f
    for f in _sources("oracle", (".py", ".c", ".h")):
        text = open(f).read()
        assert "csrc" not in text and "libc128compress" not in text, f
        assert not re.search(r"^\s*(import|from)\s+deepseek_v4_sparse_c128_gb300\.(binding|build)", text, flags=re.M), f
        assert not re.search(r"#include\s+\"[^\"]*c128(compress|_internal)", text), f


def test_inputs_module_holds_no_method_arithmetic():
    text = open(os.path.join(ROOT, "deepseek_v4_sparse_c128_gb300", "inputs.py")).read()
    for word in ("softmax", "np.exp", "rsqrt", "sqrt", "e4m3", "bfloat16", "float8", "log2", "ceil("):
        assert word not in text, word
    assert np is not None


def _ex_args(**over):
    """A valid empty batch for compress_norm_rope_store_ex: the C4 indexer FP8 layout."""
    I32, I64, F32, U8 = binding.C128_I32, binding.C128_I64, binding.C128_F32, binding.C128_U8
    a = dict(cfg=binding.config(128, 4, 1, 256, 1), ttr=_t([0], I32), pos=_t([0], I64), slot=_t([0], I64),
             bt=_t([4, 64], I32), state=_t([64, 8, 512], F32), rms=_t([128], F32), eps=1e-6, cs=_t([512, 64], F32),
             kc=_t([4, 3, 132], U8), kvs=_t([0], I64), bs=3, comp=None)
    a.update(over)
    return a


def _call_ex(L, a):
    r = lambda x: ctypes.byref(x) if x is not None else None
    return L.compress_norm_rope_store_ex(r(a["cfg"]), r(a["ttr"]), r(a["pos"]), r(a["slot"]), r(a["bt"]),
                                         r(a["state"]), r(a["rms"]), ctypes.c_float(a["eps"]), r(a["cs"]), r(a["kc"]),
                                         r(a["kvs"]), a["bs"], r(a["comp"]), None)


@pytest.mark.parametrize("case,code", [
    ("ok", 0), ("mxfp4_odd_block", 0), ("sparse_c4", 0), ("null_config", 1), ("kc_record_short", 3),
    ("comp_width", 3), ("rope32", 6), ("sparse_head128", 6), ("indexer_head512", 6), ("format9", 6),
    ("ratio3", 6), ("ratio512", 6), ("overlap2", 6), ("window_257_plus", 6), ("state_width_small", 6),
    ("state_width_odd", 6), ("state_row_mismatch", 6), ("rms_width", 6), ("fp8_stride_not_4", 5),
    ("sparse_stride_not_8", 5), ("mxfp4_stride_odd", 5),
])
def test_ex_validation_codes(L, case, code):
    """Host checks of the configurable entry point (an empty batch: nothing is launched, so a
    valid configuration returns 0 without a GPU)."""
    I32, F32, U8 = binding.C128_I32, binding.C128_F32, binding.C128_U8
    a = _ex_args()
    if case == "mxfp4_odd_block":
        a.update(cfg=binding.config(128, 4, 1, 256, 2), kc=_t([4, 3, 68], U8))
    elif case == "sparse_c4":
        a.update(cfg=binding.config(512, 4, 1, 1024, 0), state=_t([64, 8, 2048], F32), rms=_t([512], F32),
                 kc=_t([4, 3, 584], U8))
    elif case == "null_config":
        a["cfg"] = None
    elif case == "kc_record_short":
        a["kc"] = _t([4, 3, 100], U8)
    elif case == "comp_width":
        a["comp"] = _t([0, 512], F32)
    elif case == "rope32":
        c = binding.config(128, 4, 1, 256, 1)
        c.rope_head_dim = 32
        a["cfg"] = c
    elif case == "sparse_head128":
        a["cfg"] = binding.config(128, 4, 1, 256, 0)
    elif case == "indexer_head512":
        a["cfg"] = binding.config(512, 4, 1, 1024, 1)
    elif case == "format9":
        a["cfg"] = binding.config(128, 4, 1, 256, 9)
    elif case == "ratio3":
        a["cfg"] = binding.config(128, 3, 1, 256, 1)
    elif case == "ratio512":
        a["cfg"] = binding.config(128, 512, 0, 256, 1)
    elif case == "overlap2":
        a["cfg"] = binding.config(128, 4, 2, 384, 1)
    elif case == "window_257_plus":
        a["cfg"] = binding.config(128, 256, 1, 256, 1)
    elif case == "state_width_small":
        a["cfg"] = binding.config(128, 4, 1, 128, 1)
    elif case == "state_width_odd":
        a.update(cfg=binding.config(128, 4, 1, 258, 1), state=_t([64, 8, 516], F32))
    elif case == "state_row_mismatch":
        a["state"] = _t([64, 8, 1024], F32)
    elif case == "rms_width":
        a["rms"] = _t([512], F32)
    elif case == "fp8_stride_not_4":
        a["kc"] = _t([4, 1, 133], U8)
        a["bs"] = 1
    elif case == "sparse_stride_not_8":
        a.update(cfg=binding.config(512, 4, 1, 1024, 0), state=_t([64, 8, 2048], F32), rms=_t([512], F32),
                 kc=_t([4, 1, 588], U8), bs=1)
    elif case == "mxfp4_stride_odd":
        a.update(cfg=binding.config(128, 4, 1, 256, 2), kc=_t([4, 1, 69], U8), bs=1)
    assert _call_ex(L, a) == code


# ------------------------------------------------------------------ read-bandwidth probe (host side)
@pytest.mark.parametrize("args,code", [
    ((FAKE, 24, 512, 2, 8), 7),         # bytes not a multiple of 16
    ((FAKE, -16, 512, 2, 8), 7),        # negative size
    ((FAKE, 64, 48, 2, 8), 7),          # threads not a multiple of 32
    ((FAKE, 64, 2048, 1, 8), 7),        # threads above 1024
    ((FAKE, 64, 1024, 3, 8), 7),        # more than 2048 threads per SM
    ((FAKE, 64, 512, 0, 8), 7),         # no CTA per SM
    ((FAKE, 64, 512, 2, 16), 7),        # loads in flight outside 1, 2, 4, 8
    ((FAKE, 64, 512, 2, 3), 7),
    ((0, 64, 512, 2, 8), 1),            # NULL buffer
    ((FAKE + 8, 64, 512, 2, 8), 5),     # buffer not 16-byte aligned
    ((0, 0, 512, 2, 8), 0),             # empty: no-op, nothing touched
])
def test_read_probe_validation(L, args, code):
    buf, nbytes, threads, ctas, loads = args
    assert L.c128_read_probe(buf, nbytes, threads, ctas, loads, FAKE, None) == code


def test_read_probe_null_result_word(L):
    assert L.c128_read_probe(FAKE, 64, 512, 2, 8, None, None) == 1
    assert L.c128_read_probe(FAKE, 64, 512, 2, 8, FAKE + 2, None) == 5


def test_missing_library_fails_loudly(tmp_path):
    """Without the built library the binding raises at load: there is no other path to fall back
    to (run in a fresh interpreter, since this process has the library loaded already)."""
    import subprocess
    import sys
    code = ("from deepseek_v4_sparse_c128_gb300 import binding\n"
            "try:\n"
            f"    binding.load({str(tmp_path / 'libc128compress.so')!r})\n"
            "except RuntimeError as e:\n"
            "    print('raised', 'not found' in str(e))\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=root, timeout=300)
    assert out.stdout.strip() == "raised True", out.stdout + out.stderr
