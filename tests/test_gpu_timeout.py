"""The failure handling of the kernels on the GPU, without a fault: test-only entry points arm one
pipeline stage of the compress kernel, the small-window kernel or the indexer kernel and never
fill it. The bounded waits must give up, the kernel must report
C128_DEV_TIMEOUT through the device error bits and end, and the CUDA context must stay usable: the
next normal call on the same inputs matches the oracle."""
import time

import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import check_against_oracle, run_gpu, to_device

pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 32


@pytest.fixture(scope="module")
def binding():
    from deepseek_v4_sparse_c128_gb300 import binding as b
    from deepseek_v4_sparse_c128_gb300 import build
    build.build()
    b.load()
    return b


@pytest.mark.parametrize("tokens", [300, 2000])  # one CTA per token; planning pass + window queue
def test_stalled_stage_times_out_and_the_context_survives(binding, tokens):
    import torch
    p = inputs.make_problem("sweep", tokens=tokens)
    d = to_device(p)
    binding.device_errors(clear=True)
    t0 = time.monotonic()
    binding.debug_stall_first_window(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                     d["state"], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
                                     d["kv_slot_mapping"], p.kv_block_size)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    bits = binding.device_errors(clear=True)
    assert bits & TIMEOUT_BIT, bits
    assert 0.5 < waited < 20.0, waited  # the 1 s limit, not a hang
    # some windows were still stored by the CTAs that did not stall
    assert not np.array_equal(d["k_cache"].cpu().numpy(), p.k_cache)
    # the context is intact: a normal call on fresh outputs matches the oracle
    kc, comp, err = run_gpu(p)
    assert err == 0
    check_against_oracle(p, kc, comp, threads=16)


def test_stall_needs_the_compress_kernel(binding):
    p = inputs.make_problem("decode")  # 128 tokens: the cluster-split kernel
    d = to_device(p)
    with pytest.raises(binding.C128Error) as e:
        binding.debug_stall_first_window(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                         d["state"], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
                                         d["kv_slot_mapping"], p.kv_block_size)
    assert e.value.status == 7


@pytest.mark.parametrize("name", ["c4_sparse", "idx_c4_fp8", "idx_c128_mxfp4"])  # small-window x2, indexer
def test_stalled_stage_times_out_in_the_ring_kernels(binding, name):
    import torch
    from gpu_util import check_against_oracle_ex, run_gpu_ex
    p = inputs.make_next_problem(name)
    d = to_device(p)
    cfg = binding.config(p.head, p.ratio, p.overlap, p.state_width, p.fmt)
    binding.device_errors(clear=True)
    t0 = time.monotonic()
    binding.debug_stall_first_window_ex(cfg, d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                        d["state"], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
                                        d["kv_slot_mapping"], p.kv_block_size)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    bits = binding.device_errors(clear=True)
    assert bits & TIMEOUT_BIT, bits
    assert 0.5 < waited < 20.0, waited
    assert not np.array_equal(d["k_cache"].cpu().numpy(), p.k_cache)
    kc, comp, err = run_gpu_ex(p)
    assert err == 0
    check_against_oracle_ex(p, kc, comp, threads=16)
