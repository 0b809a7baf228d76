"""c128_get_info: the launch facts the library reports agree with the device and with what the
calls do (the compress kernel's shape, the planning chunk, the wait limit); and calls whose token
count sits one either side of a planning chunk boundary."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def binding():
    from deepseek_v4_sparse_c128_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def test_info_matches_the_device(binding):
    import torch
    info = binding.info()
    props = torch.cuda.get_device_properties(0)
    assert info["sm_count"] == props.multi_processor_count
    # scheduler warp, copy warp, 8 consumer warps; a 6-stage ring of 32 KiB state blocks
    assert info["threads"] == 320
    assert info["stages"] == 6
    assert 6 * 32 * 1024 <= info["smem_bytes"] <= 227 * 1024
    assert info["ctas_per_sm"] == 1  # persistent: one CTA per SM
    assert info["plan_tokens_per_cta"] == 2048
    assert info["wait_timeout_ms"] == 1000
    assert info["version"] > 0


def test_calls_around_the_chunk_size(binding):
    """Batches one token either side of a planning chunk boundary and of two chunks (the
    per-chunk lists and their counts), on the planned path, in two-level parity with the oracle."""
    from deepseek_v4_sparse_c128_gb300 import inputs
    from gpu_util import check_against_oracle, run_gpu
    chunk = binding.info()["plan_tokens_per_cta"]
    for i, T in enumerate((chunk - 1, chunk, chunk + 1, 2 * chunk + 1)):
        p = inputs.random_problem(300 + i, num_tokens=T, num_reqs=40, max_blocks=120, num_blocks=500,
                                  kv_block_size=16, active_frac=0.1)
        kc, comp, err = run_gpu(p)
        rep = check_against_oracle(p, kc, comp, threads=16)
        assert err == rep["oracle_err_bits"] == 0
        assert rep["stored"] > 0
