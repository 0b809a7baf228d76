"""The workspace of compress_norm_rope_store grows without the host waiting on the GPU.

The call is stream-ordered and asynchronous (no host synchronisation, no device-to-host read,
nothing allocated with cudaMalloc), which the CUDA-graph-captured serving path of vLLM PR #44230
relies on. A stream's workspace (claim counters, sticky error bits, token list) grows inside the
stream: pool allocation, device-to-device header copy and pool free all on the call's stream.
These tests check that a growing call returns while the stream is still busy, that the error
bits of the earlier call survive the growth, that a capture which would have to grow is refused
with C128_ERR_CAPTURE (and one that fits is captured), and that c128_release_stream returns a
stream's workspace.
"""
import time

import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import NAN_BITS, check_against_oracle, to_device

pytestmark = pytest.mark.gpu


def _call(binding, p, d, comp=None, stream=None):
    binding.compress_norm_rope_store(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                     d["state"], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
                                     d["kv_slot_mapping"], p.kv_block_size, stream=stream, comp_out=comp)


def _comp(torch, p):
    return torch.full((p.num_tokens, 512), NAN_BITS, dtype=torch.int32, device="cuda").view(torch.float32)


def _bad_block_decode():
    """The decode workload with one window's block id out of range (an error bit, no store)."""
    p = inputs.make_problem("decode")
    pos0 = int(p.positions[0])
    p.block_table[int(p.token_to_req[0]), (pos0 - 127) // 8 + 3] = p.state.shape[0] + 7
    return p


def test_growth_between_back_to_back_calls_never_waits():
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    small = _bad_block_decode()                   # 128 tokens: a 4096-token workspace
    big = inputs.make_problem("varlen16k")        # about 16k tokens: the workspace must grow
    assert big.num_tokens > 4096
    ds, db = to_device(small), to_device(big)
    # warm-up on another stream: module loading and per-device set-up happen here, not below
    warm = torch.cuda.Stream()
    _call(binding, small, to_device(small), stream=warm)
    _call(binding, big, to_device(big), stream=warm)
    torch.cuda.synchronize()
    binding.device_errors(warm, clear=True)
    binding.release_stream(warm)
    cs, cb = _comp(torch, small), _comp(torch, big)
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(int(1.5e9))             # about 0.75 s of GPU time ahead of the calls
        t0 = time.perf_counter()
        _call(binding, small, ds, comp=cs, stream=s)   # creates the stream's workspace
        _call(binding, big, db, comp=cb, stream=s)     # grows it, enqueued right behind
        host_s = time.perf_counter() - t0
        still_busy = not s.query()
    assert still_busy, "the stream finished before the calls returned: something waited on the GPU"
    assert host_s < 0.3, f"the two calls took {host_s:.3f} s on the host"
    s.synchronize()
    bits = binding.device_errors(s, clear=True)
    assert bits == 4, f"the first call's BAD_BLOCK bit did not survive the growth (bits {bits})"
    reps = [check_against_oracle(p, d["k_cache"].cpu().numpy(), c.cpu().numpy(), threads=16)
            for p, d, c in ((small, ds, cs), (big, db, cb))]
    assert reps[0]["oracle_err_bits"] == 4 and reps[0]["stored"] == small.num_tokens - 1
    assert reps[1]["oracle_err_bits"] == 0 and reps[1]["stored"] > 0
    binding.release_stream(s)


def test_capture_refuses_growth_and_captures_what_fits():
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    p = inputs.make_problem("decode")
    big = inputs.make_problem("varlen16k")
    d, dbig = to_device(p), to_device(big)
    s = torch.cuda.Stream()
    binding.reserve_workspace(p.num_tokens, s)    # 4096 tokens, fewer than big has
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        with pytest.raises(binding.C128Error) as e:
            _call(binding, big, dbig, stream=s)
        assert e.value.status == 11               # C128_ERR_CAPTURE, nothing enqueued
        with pytest.raises(binding.C128Error) as e2:
            binding.release_stream(s)             # a free would become part of the graph
        assert e2.value.status == 11
        _call(binding, p, d, stream=s)            # fits the reserved workspace
    assert np.array_equal(dbig["k_cache"].cpu().numpy(), big.k_cache)
    d["k_cache"].copy_(torch.from_numpy(p.k_cache).cuda())
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    got = d["k_cache"].cpu().numpy()
    # the same bytes as an eager call on a fresh stream (the eager path is oracle-checked elsewhere)
    de = to_device(p)
    se = torch.cuda.Stream()
    _call(binding, p, de, stream=se)
    torch.cuda.synchronize()
    assert np.array_equal(got, de["k_cache"].cpu().numpy())
    assert not np.array_equal(got, p.k_cache)
    # after capture the same stream grows eagerly and stores what the oracle stores
    cb = _comp(torch, big)
    _call(binding, big, dbig, comp=cb, stream=s)
    torch.cuda.synchronize()
    check_against_oracle(big, dbig["k_cache"].cpu().numpy(), cb.cpu().numpy(), threads=16)
    del g
    for st in (s, se):
        binding.release_stream(st)


def test_release_stream_starts_a_fresh_workspace():
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    p = _bad_block_decode()
    s = torch.cuda.Stream()
    d = to_device(p)
    _call(binding, p, d, stream=s)
    torch.cuda.synchronize()
    binding.release_stream(s)                     # the error bits go with the workspace
    assert binding.device_errors(s, clear=False) == 0
    q = inputs.make_problem("decode")
    dq = to_device(q)
    cq = _comp(torch, q)
    _call(binding, q, dq, comp=cq, stream=s)      # a new workspace, zeroed on the stream
    torch.cuda.synchronize()
    assert binding.device_errors(s, clear=True) == 0
    check_against_oracle(q, dq["k_cache"].cpu().numpy(), cq.cpu().numpy(), threads=8)
    binding.release_stream(s)
    binding.release_stream(s)                     # releasing twice is harmless
