"""Programmatic dependent launch between calls. The cluster-split and one-CTA-per-token kernels are
launched as programmatic dependents of whatever kernel precedes them on the stream and let their
own successor launch early; each waits for its predecessor to complete before it reads or writes
global memory. These tests put that order under load: back-to-back calls that write the same
cache slots (the later call's bytes must land), inputs rewritten by a torch kernel right before a
call, a torch kernel that reads the cache right after one, and both calls captured in one graph."""
import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import to_device

pytestmark = pytest.mark.gpu

SIZES = [1, 16, 128, 300, 1216]  # cluster split (S = 8, 8, 1), one CTA per token


@pytest.fixture(scope="module")
def binding():
    from deepseek_v4_sparse_c128_gb300 import binding as b
    from deepseek_v4_sparse_c128_gb300 import build
    build.build()
    b.load()
    return b


def _args(p, d, state=None):
    return (d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
            d["state"] if state is None else state, d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
            d["kv_slot_mapping"], p.kv_block_size)


def _alone(binding, p, state):
    """k_cache bytes of one call on `state` with a fresh k_cache."""
    import torch
    d = to_device(p)
    binding.compress_norm_rope_store(*_args(p, d, state))
    torch.cuda.synchronize()
    return d["k_cache"].cpu().numpy()


@pytest.mark.parametrize("T", SIZES)
def test_the_later_of_two_calls_lands(binding, T):
    import torch
    p = inputs.make_problem("sweep", tokens=T)
    d = to_device(p)
    other = inputs.draw_state(4242 + T, p.state.shape[0], "cuda")
    for _ in range(3):
        binding.compress_norm_rope_store(*_args(p, d, other))   # same slots, other values
        binding.compress_norm_rope_store(*_args(p, d))
    torch.cuda.synchronize()
    assert binding.device_errors(clear=True) == 0
    assert np.array_equal(d["k_cache"].cpu().numpy(), _alone(binding, p, d["state"]))


@pytest.mark.parametrize("T", SIZES)
def test_inputs_written_just_before_and_output_read_just_after(binding, T):
    import torch
    p = inputs.make_problem("sweep", tokens=T)
    d = to_device(p)
    final = d["state"].clone()
    d["state"].mul_(-3.0)                       # garbage state first
    binding.compress_norm_rope_store(*_args(p, d))
    d["state"].copy_(final)                     # a torch kernel rewrites the state ...
    kv = d["kv_slot_mapping"].clone()
    d["kv_slot_mapping"].fill_(-1)              # ... and parks every token, then restores them
    d["kv_slot_mapping"].copy_(kv)
    binding.compress_norm_rope_store(*_args(p, d))
    snap = d["k_cache"].clone()                 # a torch kernel reads the cache right away
    torch.cuda.synchronize()
    assert binding.device_errors(clear=True) == 0
    want = _alone(binding, p, final)
    assert np.array_equal(snap.cpu().numpy(), want)
    assert np.array_equal(d["k_cache"].cpu().numpy(), want)


@pytest.mark.parametrize("T", [16, 300])
def test_two_calls_in_one_graph(binding, T):
    import torch
    p = inputs.make_problem("sweep", tokens=T)
    d = to_device(p)
    other = inputs.draw_state(77 + T, p.state.shape[0], "cuda")
    s = torch.cuda.Stream()
    binding.reserve_workspace(T, s)
    first = binding.PreparedCall(*_args(p, d, other), stream=s)
    second = binding.PreparedCall(*_args(p, d), stream=s)
    with torch.cuda.stream(s):
        first()
        second()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            first()
            second()
    d["k_cache"].copy_(torch.from_numpy(p.k_cache))
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert binding.device_errors(s, clear=True) == 0
    assert np.array_equal(d["k_cache"].cpu().numpy(), _alone(binding, p, d["state"]))
    s.synchronize()
    binding.release_stream(s)


@pytest.mark.parametrize("head,ratio,overlap,fmt", [(512, 4, 1, 0), (128, 4, 1, 1), (128, 4, 1, 2), (128, 128, 0, 1)])
def test_the_later_of_two_calls_lands_other_configurations(binding, head, ratio, overlap, fmt):
    """The small-window and indexer kernels in their token-striding range (at most 8 tokens per
    SM), launched the same way: two calls on the same slots back to back, the later one's bytes."""
    import torch
    p = inputs.prefill_problem("pdl", 3, 3, 5 if ratio == 4 else 128, 300 if ratio == 4 else 500, head, ratio,
                               overlap, fmt)
    assert p.num_tokens <= 8 * 148
    cfg = binding.config(p.head, p.ratio, p.overlap, p.state_width, p.fmt)

    def run(d, state, reps):
        for _ in range(reps):
            binding.compress_norm_rope_store_ex(cfg, *_args(p, d, state))

    d = to_device(p)
    other = torch.randn_like(d["state"])
    for _ in range(3):
        run(d, other, 1)
        run(d, None, 1)
    torch.cuda.synchronize()
    assert binding.device_errors(clear=True) == 0
    ref = to_device(p)
    run(ref, None, 1)
    torch.cuda.synchronize()
    assert not np.array_equal(ref["k_cache"].cpu().numpy(), p.k_cache)
    assert np.array_equal(d["k_cache"].cpu().numpy(), ref["k_cache"].cpu().numpy())
