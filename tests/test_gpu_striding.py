"""The C128 calls with more tokens than SMs and at most 8 per SM (one CTA per token, two per SM,
with no planning pass): few active windows among many tokens (most CTAs find nothing), calls
enqueued back to back on one stream with different active sets, and bad indices followed by a
clean call on the same stream; and a batch beyond the per-chunk planning pass's range."""
import numpy as np
import pytest

import oracle
from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import NAN_BITS, check_against_oracle, run_gpu, to_device, written_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_v4_sparse_c128_gb300 import build, binding
    build.build()
    binding.load()


def keep_active(p, keep):
    """Only the tokens in `keep` stay active (the others lose their state slot)."""
    mask = np.zeros(p.num_tokens, bool)
    mask[np.asarray(keep, dtype=np.int64)] = True
    p.slot_mapping[~mask] = -1
    return p


@pytest.mark.parametrize("T,active", [(300, 1), (600, 3), (1000, 10), (1216, 37), (700, 152), (1200, 600)])
def test_few_active_windows_among_many_tokens(T, active):
    """`active` windows among T tokens at random places: from one CTA with work to all of them."""
    rng = np.random.default_rng(T + active)
    p = keep_active(inputs.make_problem("sweep", tokens=T), np.sort(rng.choice(T, active, replace=False)))
    kc, comp, err = run_gpu(p)
    assert err == 0
    rep = check_against_oracle(p, kc, comp, threads=16)
    assert rep["stored"] == active


def test_calls_back_to_back_reuse_the_counters():
    """Three calls enqueued on one stream with no synchronisation in between, with different
    active sets, each against the oracle."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    rng = np.random.default_rng(5)
    base = inputs.make_problem("sweep", tokens=900)
    probs = [keep_active(inputs.make_problem("sweep", tokens=900), np.sort(rng.choice(900, n, replace=False)))
             for n in (900, 77, 400)]
    runs = []
    for p in probs:
        dev = to_device(p)
        comp = torch.full((p.num_tokens, 512), NAN_BITS, dtype=torch.int32, device="cuda").view(torch.float32)
        runs.append((p, dev, comp))
    for p, dev, comp in runs:
        binding.compress_norm_rope_store(dev["token_to_req"], dev["positions"], dev["slot_mapping"],
                                         dev["block_table"], dev["state"], dev["rms_w"], p.eps, dev["cos_sin"],
                                         dev["k_cache"], dev["kv_slot_mapping"], p.kv_block_size, comp_out=comp)
    torch.cuda.synchronize()
    assert binding.device_errors(clear=True) == 0
    for p, dev, comp in runs:
        rep = check_against_oracle(p, dev["k_cache"].cpu().numpy(), comp.cpu().numpy(), threads=16)
        assert rep["stored"] == int((p.slot_mapping >= 0).sum())
    assert base.num_tokens == 900


def test_bad_indices_then_a_clean_call():
    """Three active windows, one with a bad block id and one with a bad kv slot: those two store
    nothing and report their bits, the third is stored; the next call on the same stream (all
    windows good) matches the oracle."""
    p = keep_active(inputs.make_problem("sweep", tokens=500), [17, 250, 499])
    first = (int(p.positions[250]) - 127) // 8
    p.block_table[int(p.token_to_req[250]), first + 13] = p.state.shape[0]  # BAD_BLOCK
    p.kv_slot_mapping[499] = p.k_cache.shape[0] * p.kv_block_size          # BAD_KV_SLOT
    kc, comp, err = run_gpu(p)
    ref = p.k_cache.copy()
    assert err == oracle.forward(p, k_cache=ref) == (4 | 16)
    rep = check_against_oracle(p, kc, comp)
    assert rep["stored"] == 1 and written_rows(comp).tolist() == [17]
    q = keep_active(inputs.make_problem("sweep", tokens=500), [17, 250, 499])
    kc, comp, err = run_gpu(q)
    assert err == 0
    assert check_against_oracle(q, kc, comp)["stored"] == 3


def test_more_tokens_than_the_per_chunk_plan_covers():
    """Above 512 x 2048 tokens the planning pass falls back to one compact list behind a zeroing
    pass: the mixed workload padded with inactive tokens to 1,048,577 tokens."""
    import dataclasses
    p = inputs.make_problem("mixed")
    T = 512 * 2048 + 1
    pad = T - p.num_tokens
    q = dataclasses.replace(
        p, token_to_req=np.concatenate([p.token_to_req, np.zeros(pad, np.int32)]),
        positions=np.concatenate([p.positions, np.full(pad, 127, np.int64)]),
        slot_mapping=np.concatenate([p.slot_mapping, np.full(pad, -1, np.int64)]),
        kv_slot_mapping=np.concatenate([p.kv_slot_mapping, np.zeros(pad, np.int64)]))
    kc, comp, err = run_gpu(q, comp=False)
    assert err == 0
    ref = q.k_cache.copy()
    oracle.forward(q, k_cache=ref, threads=16)
    from gpu_util import slots_agree
    rows = np.nonzero((q.slot_mapping >= 0) & ((q.positions + 1) % 128 == 0) & (q.kv_slot_mapping >= 0))[0]
    assert rows.size > 10
    differ, _, _ = slots_agree(q, kc, ref, rows)
    assert differ <= 2  # rounding ties only
