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
        out.update(e2e_bytes_differ=int(d2.sum()), e2e_windows_differ=bad_windows,
                   fp8_codes_differ=int(sum(d2[slot_ranges(problem, t)[0]][:448].sum() for t in rows_ref)))
    return out
