"""Helpers shared by the GPU parity tests: move a Problem to the device, run the CUDA path, and
build the expected bytes from the oracle."""
from __future__ import annotations

import numpy as np

import oracle

TOL_ABS, TOL_REL = 1e-6, 1e-5   # fp32 compressed vector vs the oracle (binary64 softmax)
NAN_BITS = 0x7FC00001           # sentinel for comp rows that were not written


def to_device(problem, device="cuda"):
    import torch
    d = {}
    for name in ("token_to_req", "positions", "slot_mapping", "block_table", "rms_w", "cos_sin", "k_cache",
                 "kv_slot_mapping"):
        d[name] = torch.from_numpy(np.ascontiguousarray(getattr(problem, name))).to(device)
    st = problem.state
    d["state"] = st if hasattr(st, "is_cuda") else torch.from_numpy(st).to(device)
    return d


def run_gpu(problem, dev=None, comp=True, stream=None):
    """Run the CUDA op; returns (k_cache bytes as numpy, comp32 [T,512] numpy or None, device errors)."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    dev = dev or to_device(problem)
    T = problem.num_tokens
    comp_out = None
    if comp:
        comp_out = torch.full((T, 512), 0, dtype=torch.int32, device=dev["state"].device)
        comp_out.fill_(NAN_BITS)
        comp_out = comp_out.view(torch.float32)
    binding.compress_norm_rope_store(dev["token_to_req"], dev["positions"], dev["slot_mapping"], dev["block_table"],
                                     dev["state"], dev["rms_w"], problem.eps, dev["cos_sin"], dev["k_cache"],
                                     dev["kv_slot_mapping"], problem.kv_block_size, stream=stream, comp_out=comp_out)
    torch.cuda.synchronize()
    err = binding.device_errors(stream, clear=True)
    kc = dev["k_cache"].cpu().numpy()
    cp = comp_out.cpu().numpy() if comp_out is not None else None
    return kc, cp, err


def written_rows(comp: np.ndarray) -> np.ndarray:
    return np.nonzero(~np.all(comp.view(np.uint32) == NAN_BITS, axis=1))[0]


def slot_ranges(problem, t):
    """Byte ranges (token data, scales) of token t's kv slot in the flattened k_cache (the
    cache-block layout of the fused_compress_quant_cache API page)."""
    s = int(problem.kv_slot_mapping[t])
    bs = problem.kv_block_size
    stride = problem.k_cache.shape[1] * problem.k_cache.shape[2]
    blk, off = divmod(s, bs)
    tok = blk * stride + off * 576
    scl = blk * stride + bs * 576 + off * 8
    return slice(tok, tok + 576), slice(scl, scl + 8)


def replay_expected(problem, comp: np.ndarray, rows) -> np.ndarray:
    """k_cache expected when the oracle's epilogue is applied to the given comp32 rows."""
    kc = problem.k_cache.copy()
    flat = kc.reshape(-1)
    for t in rows:
        p = int(problem.positions[t])
        tok, sc = oracle.epilogue(comp[t], problem.rms_w, problem.eps, problem.cos_sin[(p // 128) * 128])
        a, b = slot_ranges(problem, t)
        flat[a] = tok
        flat[b] = sc
    return kc


def comp_close(gpu: np.ndarray, ref: np.ndarray):
    """(ok, max abs err, max err / tolerance) of gpu vs ref comp32 rows."""
    g, r = gpu.astype(np.float64), ref.astype(np.float64)
    err = np.abs(g - r)
    tol = TOL_ABS + TOL_REL * np.abs(r)
    return bool(np.all(err <= tol)), float(err.max(initial=0.0)), float((err / tol).max(initial=0.0))


def check_against_oracle(problem, kc_gpu, comp_gpu, threads=8, tokens=None):
    """Two-level parity. Returns a dict of counts; asserts the parts that must hold exactly."""
    T = problem.num_tokens
    comp_ref = np.full((T, 512), np.nan, np.float32)
    comp_ref.view(np.uint32)[:] = NAN_BITS
    kc_ref = problem.k_cache.copy()
    err_ref = oracle.forward(problem, k_cache=kc_ref, comp_out=comp_ref, threads=threads, tokens=tokens)
    rows_ref = written_rows(comp_ref)
    rows_gpu = written_rows(comp_gpu)
    if tokens is not None:
        rows_gpu = np.intersect1d(rows_gpu, np.asarray(tokens))
    assert np.array_equal(rows_ref, rows_gpu), "the set of stored tokens differs from the oracle's"
    ok, max_abs, worst = comp_close(comp_gpu[rows_ref], comp_ref[rows_ref])
    assert ok, f"compressed vector outside 1e-6 + 1e-5|x|: max abs {max_abs:.3g}, worst/tol {worst:.3g}"
    out = {"stored": int(rows_ref.size), "comp_max_abs": max_abs, "comp_worst_over_tol": worst,
           "oracle_err_bits": err_ref}
    if tokens is None:
        # (i) epilogue exact: the oracle's epilogue on the GPU's comp32 reproduces every byte
        kc_replay = replay_expected(problem, comp_gpu, rows_ref)
        diff = np.nonzero(kc_replay.reshape(-1) != kc_gpu.reshape(-1))[0]
        assert diff.size == 0, f"{diff.size} bytes differ from the oracle epilogue replay (first at {diff[:8]})"
        # (ii) end to end against the oracle's own comp32: differences only where comp32 differs
        d2 = kc_ref.reshape(-1) != kc_gpu.reshape(-1)
        bad_windows = 0
        for t in rows_ref:
            a, b = slot_ranges(problem, t)
            if d2[a].any() or d2[b].any():
                bad_windows += 1
                assert not np.array_equal(comp_gpu[t].view(np.uint32), comp_ref[t].view(np.uint32))
        _, max_deq, max_rope = slots_agree(problem, kc_gpu, kc_ref, rows_ref)
        out.update(e2e_bytes_differ=int(d2.sum()), e2e_windows_differ=bad_windows,
                   fp8_codes_differ=int(sum(d2[slot_ranges(problem, t)[0]][:448].sum() for t in rows_ref)),
                   max_dequant_diff=max_deq, max_rope_diff=max_rope)
    return out


# --------------------------------------------------------------- byte-level agreement of two runs
def _e4m3_table() -> np.ndarray:
    """Value of every e4m3fn byte from the format definition (bias 7, 3 mantissa bits)."""
    out = np.zeros(256)
    for c in range(256):
        E, m = (c >> 3) & 15, c & 7
        v = (m / 8.0) * 2.0 ** -6 if E == 0 else (1 + m / 8.0) * 2.0 ** (E - 7)
        out[c] = -v if c & 0x80 else v
    out[0x7F] = out[0xFF] = np.nan
    return out


E4M3 = _e4m3_table()


def _e4m3_step(y):
    """Spacing of e4m3 codes around magnitude y (code space)."""
    a = np.abs(y)
    return np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3))


def slots_agree(problem, kc_a, kc_b, rows):
    """Two runs of the op whose compressed vectors differ only by rounding: every byte outside
    the stored slots is identical; inside them, scale bytes differ by at most 1 and every
    dequantised nope value (e4m3 x 2^(scale-127)) by at most one quantisation step and every rope
    value (bf16) by one bf16 step plus 1e-4 (the rotation can cancel). Returns (slots that differ, max dequant diff, max rope diff), the
    quantities the pages report when they validate a kernel against another (PR #44230,
    Validation)."""
    fa, fb = kc_a.reshape(-1), kc_b.reshape(-1)
    inside = np.zeros(fa.size, bool)
    differ, max_deq, max_rope = 0, 0.0, 0.0
    for t in rows:
        tok, sc = slot_ranges(problem, t)
        inside[tok] = True
        inside[sc] = True
        if np.array_equal(fa[tok], fb[tok]) and np.array_equal(fa[sc], fb[sc]):
            continue
        differ += 1
        sa, sb = fa[sc].astype(int), fb[sc].astype(int)
        assert sa[7] == sb[7] == 0 and np.all(np.abs(sa[:7] - sb[:7]) <= 1), (t, sa, sb)
        ya = E4M3[fa[tok][:448]].reshape(7, 64)
        yb = E4M3[fb[tok][:448]].reshape(7, 64)
        pa = 2.0 ** (sa[:7] - 127.0)[:, None]
        pb = 2.0 ** (sb[:7] - 127.0)[:, None]
        va, vb = ya * pa, yb * pb
        tol = np.maximum(_e4m3_step(ya) * pa, _e4m3_step(yb) * pb) * 1.001
        d = np.abs(va - vb)
        assert np.all(d <= tol), (t, float(d.max()))
        max_deq = max(max_deq, float(d.max()))
        ra = (fa[tok][448:].view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        rb = (fb[tok][448:].view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        dr = np.abs(ra - rb)
        # one bf16 step of the output, plus an absolute 1e-4 for cancellation in e*C - o*S: the
        # inputs are O(1) after RMSNorm and move by about 1e-5 relative when comp does
        tol_r = np.maximum(np.abs(ra), np.abs(rb)) * 2.0 ** -7 + 1e-4
        assert np.all(dr <= tol_r), (t, float(dr.max()))
        max_rope = max(max_rope, float(dr.max()))
    assert np.array_equal(fa[~inside], fb[~inside]), "bytes outside the stored slots differ"
    return differ, max_deq, max_rope


# ------------------------------------------------------------ other configurations (the _ex call)
FORMAT_BYTES = {0: (576, 8), 1: (128, 4), 2: (64, 4)}


def run_gpu_ex(problem, dev=None, comp=True, stream=None):
    """Run compress_norm_rope_store_ex with the problem's configuration."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    dev = dev or to_device(problem)
    T, head = problem.num_tokens, problem.head
    comp_out = None
    if comp:
        comp_out = torch.full((T, head), NAN_BITS, dtype=torch.int32, device=dev["state"].device).view(torch.float32)
    cfg = binding.config(problem.head, problem.ratio, problem.overlap, problem.state_width, problem.fmt)
    binding.compress_norm_rope_store_ex(cfg, dev["token_to_req"], dev["positions"], dev["slot_mapping"],
                                        dev["block_table"], dev["state"], dev["rms_w"], problem.eps, dev["cos_sin"],
                                        dev["k_cache"], dev["kv_slot_mapping"], problem.kv_block_size, stream=stream,
                                        comp_out=comp_out)
    torch.cuda.synchronize()
    err = binding.device_errors(stream, clear=True)
    return dev["k_cache"].cpu().numpy(), (comp_out.cpu().numpy() if comp else None), err


def slot_ranges_ex(problem, t):
    tb, sb = FORMAT_BYTES[problem.fmt]
    s = int(problem.kv_slot_mapping[t])
    bs = problem.kv_block_size
    stride = problem.k_cache.shape[1] * problem.k_cache.shape[2]
    blk, off = divmod(s, bs)
    tok = blk * stride + off * tb
    scl = blk * stride + bs * tb + off * sb
    return slice(tok, tok + tb), slice(scl, scl + sb)


def replay_expected_ex(problem, comp, rows):
    kc = problem.k_cache.copy()
    flat = kc.reshape(-1)
    for t in rows:
        p = int(problem.positions[t])
        row = problem.cos_sin[(p // problem.ratio) * problem.ratio]
        if problem.fmt == 0:
            tok, sc = oracle.epilogue(comp[t], problem.rms_w, problem.eps, row)
        else:
            tok, sc = oracle.epilogue_indexer(problem.fmt, comp[t], problem.rms_w, problem.eps, row)
        a, b = slot_ranges_ex(problem, t)
        flat[a] = tok
        flat[b] = sc
    return kc


def check_against_oracle_ex(problem, kc_gpu, comp_gpu, threads=8):
    """Two-level parity for any configuration: same stored tokens as the oracle, comp32 within
    1e-6 + 1e-5|x|, and every k_cache byte equal to the oracle epilogue replayed on the GPU's
    comp32; bytes that differ from the oracle's own output are counted."""
    T, head = problem.num_tokens, problem.head
    comp_ref = np.zeros((T, head), np.float32)
    comp_ref.view(np.uint32)[:] = NAN_BITS
    kc_ref = problem.k_cache.copy()
    err_ref = oracle.forward_ex(problem, k_cache=kc_ref, comp_out=comp_ref, threads=threads)
    rows_ref, rows_gpu = written_rows(comp_ref), written_rows(comp_gpu)
    assert np.array_equal(rows_ref, rows_gpu), "the set of stored tokens differs from the oracle's"
    ok, max_abs, worst = comp_close(comp_gpu[rows_ref], comp_ref[rows_ref])
    assert ok, f"compressed vector outside 1e-6 + 1e-5|x|: max abs {max_abs:.3g}, worst/tol {worst:.3g}"
    kc_replay = replay_expected_ex(problem, comp_gpu, rows_ref)
    diff = np.nonzero(kc_replay.reshape(-1) != kc_gpu.reshape(-1))[0]
    assert diff.size == 0, f"{diff.size} bytes differ from the oracle epilogue replay (first at {diff[:8]})"
    d2 = kc_ref.reshape(-1) != kc_gpu.reshape(-1)
    windows = 0
    for t in rows_ref:
        a, b = slot_ranges_ex(problem, t)
        if d2[a].any() or d2[b].any():
            windows += 1
            assert not np.array_equal(comp_gpu[t].view(np.uint32), comp_ref[t].view(np.uint32))
    return {"stored": int(rows_ref.size), "comp_max_abs": max_abs, "comp_worst_over_tol": worst,
            "oracle_err_bits": err_ref, "e2e_bytes_differ": int(d2.sum()), "e2e_windows_differ": windows}
