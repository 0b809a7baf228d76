"""The entry point that allocates no device memory, c128_compress_norm_rope_store_noalloc.

It serves callers that may not call cudaMalloc once they are running (for example a serving
engine that gives all free device memory to its caches at start-up, or code inside an
allocator callback): its scratch is a static device array of C128_NOALLOC_MAX_TOKENS tokens
instead of the workspace compress_norm_rope_store allocates. These tests call it through the
C-ABI and check that two calls in a row produce exactly the k_cache bytes that the allocating
entry point produces on the same inputs (bytes are compared exactly, as everywhere in these
tests), and that a batch larger than the static array is refused without launching anything.
This file is collected last so that a run stopping at its first failure has run every other test.
"""
import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def binding():
    from deepseek_v4_sparse_c128_gb300 import binding as b
    from deepseek_v4_sparse_c128_gb300 import build
    build.build()
    b.load()
    return b


def _device(problem):
    import torch
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(problem, k))).cuda()
         for k in ("token_to_req", "positions", "slot_mapping", "block_table", "rms_w", "cos_sin", "k_cache",
                   "kv_slot_mapping")}
    d["state"] = torch.from_numpy(problem.state).cuda()
    return d


def _args(p, d):
    return (d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"], d["state"], d["rms_w"], p.eps,
            d["cos_sin"], d["k_cache"], d["kv_slot_mapping"], p.kv_block_size)


def test_noalloc_matches_the_allocating_entry_point(binding):
    import torch
    # two calls in a row on different batches (the second one starts from what the first left
    # in the shared static array), then the first batch again
    for name in ("decode", "varlen16k", "decode"):
        p = inputs.make_problem(name)
        ref, new = _device(p), _device(p)
        binding.compress_norm_rope_store(*_args(p, ref))
        binding.compress_norm_rope_store_noalloc(*_args(p, new))
        torch.cuda.synchronize()
        want = ref["k_cache"].cpu().numpy()
        got = new["k_cache"].cpu().numpy()
        assert not np.array_equal(want, p.k_cache)           # something was stored
        assert np.array_equal(got, want), name


def test_noalloc_refuses_batches_beyond_its_static_array(binding):
    import torch
    T = binding.NOALLOC_MAX_TOKENS + 1
    p = inputs.random_problem(5, num_tokens=T, num_reqs=4, max_blocks=32, num_blocks=16, kv_block_size=2)
    d = _device(p)
    with pytest.raises(binding.C128Error) as e:
        binding.compress_norm_rope_store_noalloc(*_args(p, d))
    assert e.value.status == 10
    torch.cuda.synchronize()
    assert np.array_equal(d["k_cache"].cpu().numpy(), p.k_cache)


def test_noalloc_allocates_nothing_and_covers_one_cta_per_token(binding):
    """After one warm-up call (the first call on a device loads the library's static array and
    looks up its address), two more calls on a stream the allocating entry point never used leave
    the device's free memory and torch's reserved memory exactly as they were. The batch has twice
    as many tokens as the GPU has SMs, which runs one CTA per token (two per SM)."""
    import torch
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    p = inputs.make_problem("sweep", tokens=2 * sm)
    ref, new, warm = _device(p), _device(p), _device(p)
    binding.compress_norm_rope_store(*_args(p, ref))
    binding.compress_norm_rope_store_noalloc(*_args(p, warm))
    torch.cuda.synchronize()
    want = ref["k_cache"].cpu().numpy()
    assert np.array_equal(warm["k_cache"].cpu().numpy(), want)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    for _ in range(2):
        binding.compress_norm_rope_store_noalloc(*_args(p, new), stream=s)
    torch.cuda.synchronize()
    free1, reserved1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    assert free1 == free0, f"device free memory changed by {free1 - free0} bytes"
    assert reserved1 == reserved0
    assert np.array_equal(new["k_cache"].cpu().numpy(), want)
