"""Seeded random configurations of compress_norm_rope_store_ex against the oracle: cache format,
compress ratio (1..256), overlap, state block size (1..64), kv block size (odd ones included),
request count and lengths, decode tails. Each case takes whichever kernel its configuration
selects (small-window ring, tiled or per-row copies; indexer ring; gather) and must pass the
two-level parity."""
import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import check_against_oracle_ex, run_gpu_ex

pytestmark = pytest.mark.gpu


def _case(i: int):
    rng = np.random.default_rng([2026, i])
    fmt = int(rng.integers(0, 3))
    head = 512 if fmt == 0 else 128
    while True:
        ratio = int(2 ** rng.integers(0, 9))
        overlap = int(rng.integers(0, 2))
        if (1 + overlap) * ratio <= 256:
            break
    return dict(fmt=fmt, head=head, ratio=ratio, overlap=overlap, sblk=int(rng.choice([1, 2, 4, 8, 16, 32, 64])),
                kvbs=int(rng.choice([1, 3, 16, 64])), reqs=int(rng.integers(1, 10)), maxlen=int(rng.integers(1, 1500)),
                tail=int(rng.integers(0, 30)), seed=int(rng.integers(1 << 30)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_v4_sparse_c128_gb300 import binding, build
    build.build()
    binding.load()


@pytest.mark.parametrize("i", range(48))
def test_random_configuration(i):
    c = _case(i)
    p = inputs.prefill_problem("fuzz", c["seed"], c["reqs"], 1, c["maxlen"], c["head"], c["ratio"], c["overlap"],
                               c["fmt"], state_block=c["sblk"], kv_block_size=c["kvbs"], decode_tail=c["tail"])
    kc, comp, err = run_gpu_ex(p)
    assert err == 0, c
    check_against_oracle_ex(p, kc, comp, threads=16)
