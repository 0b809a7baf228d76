"""Seeded random configurations against the oracle.

compress_norm_rope_store_ex: cache format, compress ratio (1..256), overlap, state block size
(1..64), kv block size (odd ones included), request count and lengths, decode tails; each case
takes whichever kernel its configuration selects (small-window ring with tiled or per-row copies,
indexer ring, gather). compress_norm_rope_store: random batches of 1..5000 tokens over its three
call paths (cluster split, one CTA per token, planning pass), with aliased blocks, padded tokens,
negative positions and missing kv slots. On half the cases a few tokens get out-of-range
request rows, block ids, block-table columns or kv slots: the device error bits and the stored
set must then equal the oracle's. Every case passes the two-level parity.

C128_FUZZ_ROUNDS=k (environment) runs k times as many cases of both generators (new seeds
after the default ones), for soak runs."""
import os

import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import check_against_oracle, check_against_oracle_ex, run_gpu, run_gpu_ex

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_v4_sparse_c128_gb300 import binding, build
    build.build()
    binding.load()


def _plant(p, seed: int, window_rows: int, ratio: int):
    """Out-of-range indices on about 2 % of the tokens."""
    rng = np.random.default_rng(seed)
    T, B = p.num_tokens, p.state.shape[1]
    for t in rng.choice(T, size=max(1, T // 50), replace=False):
        what = int(rng.integers(0, 4))
        if what == 0:
            p.token_to_req[t] = p.block_table.shape[0] + int(rng.integers(0, 3))
        elif what == 1:
            r = int(p.token_to_req[t])
            if 0 <= r < p.block_table.shape[0] and p.positions[t] >= 0:
                q = int(p.positions[t]) - int(rng.integers(0, window_rows))
                if q >= 0 and q // B < p.block_table.shape[1]:
                    p.block_table[r, q // B] = p.state.shape[0] + int(rng.integers(0, 5))
        elif what == 2:
            p.kv_slot_mapping[t] = p.k_cache.shape[0] * p.kv_block_size + int(rng.integers(0, 5))
        else:
            p.positions[t] = p.block_table.shape[1] * B + ratio * int(rng.integers(0, 3)) + ratio - 1


def _case_ex(i: int):
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


_ROUNDS = max(1, int(os.environ.get("C128_FUZZ_ROUNDS", "1")))


@pytest.mark.parametrize("i", range(48 * _ROUNDS))
def test_random_configuration(i):
    c = _case_ex(i)
    p = inputs.prefill_problem("fuzz", c["seed"], c["reqs"], 1, c["maxlen"], c["head"], c["ratio"], c["overlap"],
                               c["fmt"], state_block=c["sblk"], kv_block_size=c["kvbs"], decode_tail=c["tail"])
    if i % 2 and p.num_tokens:
        _plant(p, c["seed"] + 1, (1 + c["overlap"]) * c["ratio"], c["ratio"])
    kc, comp, err = run_gpu_ex(p)
    rep = check_against_oracle_ex(p, kc, comp, threads=16)
    assert err == rep["oracle_err_bits"], (c, err, rep["oracle_err_bits"])
    if i % 2 == 0:
        assert err == 0, c


@pytest.mark.parametrize("i", range(32 * _ROUNDS))
def test_random_c128_batch(i):
    rng = np.random.default_rng([128, i])
    T = int(rng.choice([int(rng.integers(1, 160)), int(rng.integers(150, 1300)), int(rng.integers(1200, 5000))]))
    seed = int(rng.integers(1 << 30))
    p = inputs.random_problem(seed, num_tokens=T, num_reqs=int(rng.integers(1, 64)),
                              max_blocks=int(rng.integers(17, 200)), num_blocks=int(rng.integers(16, 600)),
                              kv_block_size=int(rng.choice([1, 2, 3, 16, 64])),
                              active_frac=float(rng.choice([0.1, 0.5, 0.95])))
    if i % 2:
        _plant(p, seed + 1, 128, 128)
    kc, comp, err = run_gpu(p)
    rep = check_against_oracle(p, kc, comp, threads=16)
    assert err == rep["oracle_err_bits"], (T, err, rep["oracle_err_bits"])
