"""Long contexts: window ends spread up to position 1,048,575 (a block table of 131,088 columns, a
cos/sin cache of 1,048,704 rows), so the window start, the block-table column, the cos/sin row and
every address built from them are far past the ranges of the other workloads.
- C128: one case per launch mode, cluster split (100 tokens), one CTA per token (300), planning pass
  and window queue (2000); random requests, padded tokens, negative positions and missing kv
  slots as in the other random problems.
- The other configurations (C4 sparse, C4 indexer FP8 and MXFP4, ratio-128 indexer): one-token
  requests near position 1,048,575, in the token-striding range and, behind 1500 padded tokens,
  on the planning path."""
import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu

MAX_BLOCKS = (1 << 20) // 8 + 16  # positions up to 1,048,703


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_v4_sparse_c128_gb300 import build, binding
    build.build()
    binding.load()


@pytest.mark.parametrize("T", [100, 300, 2000])
def test_positions_near_one_million(T):
    p = inputs.random_problem(4000 + T, num_tokens=T, num_reqs=5, max_blocks=MAX_BLOCKS, num_blocks=300,
                              kv_block_size=2, active_frac=0.7)
    active = (p.slot_mapping >= 0) & (p.positions >= 0) & ((p.positions + 1) % 128 == 0) & (p.kv_slot_mapping >= 0)
    assert int(p.positions[active].max()) > 900_000  # the case reaches far positions
    kc, comp, err = run_gpu(p)
    assert err == 0
    rep = check_against_oracle(p, kc, comp, threads=16)
    assert rep["stored"] == int(active.sum())


# ------------------------------------------------ the other configurations (compress_norm_rope_store_ex)
@pytest.fixture(scope="module")
def far_cos_sin():
    return inputs._cos_sin_cache(MAX_BLOCKS * 8)


def far_decode_problem(seed, head, ratio, overlap, fmt, cos_sin, num_reqs=24, pad_tokens=0, kv_block_size=2):
    """One-token requests at window ends near position 1,048,575; block tables of 131,088 columns
    with iid block ids from a small pool (windows alias blocks); `pad_tokens` padded tokens
    (slot -1) in front push the batch onto the planning path."""
    rng = np.random.default_rng([seed, head, ratio, fmt])
    sw = head * (1 + overlap)
    nb = 512
    k = rng.integers((1 << 20) // ratio - 900, (1 << 20) // ratio, size=num_reqs)
    pos_act = (ratio * k - 1).astype(np.int64)
    bt = rng.integers(0, nb, size=(num_reqs, MAX_BLOCKS)).astype(np.int32)
    req = np.concatenate([np.zeros(pad_tokens, np.int32), np.arange(num_reqs, dtype=np.int32)])
    pos = np.concatenate([rng.integers(0, 1 << 20, size=pad_tokens).astype(np.int64), pos_act])
    slot = np.concatenate([np.full(pad_tokens, -1, np.int64), np.ones(num_reqs, np.int64)])
    nkb = -(-num_reqs // kv_block_size)
    kv_slot = np.concatenate([np.full(pad_tokens, -1, np.int64),
                              rng.permutation(nkb * kv_block_size)[:num_reqs].astype(np.int64)])
    return inputs.Problem(f"far{seed}", req, pos, slot, bt, inputs.draw_state_rows(seed, nb, 8, sw, "cpu"),
                          inputs._rms_w(rng)[:head].copy(), 1e-6, cos_sin,
                          rng.integers(0, 256, size=(nkb, kv_block_size, inputs.SLOT_BYTES[fmt]), dtype=np.uint8),
                          kv_slot, kv_block_size, head=head, ratio=ratio, overlap=overlap, state_width=sw, fmt=fmt)


@pytest.mark.parametrize("pad", [0, 1500])
@pytest.mark.parametrize("head,ratio,overlap,fmt", [(512, 4, 1, 0), (128, 4, 1, 1), (128, 4, 1, 2), (128, 128, 0, 1)])
def test_other_configurations_near_one_million(far_cos_sin, head, ratio, overlap, fmt, pad):
    from gpu_util import check_against_oracle_ex, run_gpu_ex
    p = far_decode_problem(7 + pad, head, ratio, overlap, fmt, far_cos_sin, pad_tokens=pad)
    kc, comp, err = run_gpu_ex(p)
    assert err == 0
    rep = check_against_oracle_ex(p, kc, comp)
    assert rep["stored"] == 24
