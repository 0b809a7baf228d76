"""Extreme scores through the whole path, against the oracle (two-level parity):
- -inf scores on random rows of random columns (never a whole column): those rows get weight 0,
  as in a masked softmax;
- scores scaled by 1e4: nearly one-hot weights, where exp(s - max) underflows for all but the top
  rows and nothing may overflow;
- scores offset by +1e4 or -1e4 per state block: large magnitudes, where within a window the
  blocks with the lower offset get weights that underflow to 0.
Each on every C128 call path (cluster split, one CTA per token, planning pass); and -inf scores in
the four other configurations."""
import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_v4_sparse_c128_gb300 import build, binding
    build.build()
    binding.load()


def _scores(p):
    return p.state[:, :, 512:]  # [NB, 8, 512] view of the score half of every row


@pytest.mark.parametrize("T", [100, 300, 2000])
@pytest.mark.parametrize("kind", ["neg_inf_rows", "peaked", "shifted"])
def test_extreme_scores(T, kind):
    p = inputs.make_problem("sweep", tokens=T)
    rng = np.random.default_rng([T, len(kind)])
    sc = _scores(p)
    if kind == "neg_inf_rows":
        # every state row belongs to exactly one window here, so at most 8 of a block's rows and
        # never all 128 rows of a window lose a column
        mask = rng.random(sc.shape) < 0.3
        mask[:, 0, :] = False  # row 0 of every block keeps every column finite
        sc[mask] = -np.inf
    elif kind == "peaked":
        sc *= np.float32(1e4)
    else:
        sc += np.float32(1e4) * np.where(rng.random((sc.shape[0], 1, 1)) < 0.5, -1, 1).astype(np.float32)
    kc, comp, err = run_gpu(p)
    assert err == 0
    rep = check_against_oracle(p, kc, comp, threads=16)
    assert rep["stored"] == T
    assert np.isfinite(comp[np.isfinite(comp[:, 0])]).all()


@pytest.mark.parametrize("name", ["c4_sparse", "idx_c4_fp8", "idx_c4_mxfp4", "idx_c128_fp8"])
def test_neg_inf_scores_other_configurations(name):
    """-inf scores on random columns of random rows, except the last row of every group of
    `ratio` positions, so every window keeps a finite score in each column (with overlap the older
    group's last row is the finite one of its half)."""
    from gpu_util import check_against_oracle_ex, run_gpu_ex
    p = inputs.make_next_problem(name, scale=1)
    rng = np.random.default_rng(len(name))
    sw, sb = p.state_width, p.state.shape[1]
    for r in range(p.block_table.shape[0]):
        qs = p.positions[p.token_to_req == r]
        for q in qs[(qs >= 0) & (qs % p.ratio != p.ratio - 1)]:
            if rng.random() < 0.3:
                cols = rng.random(sw) < 0.5
                p.state[p.block_table[r, q // sb], q % sb, sw:][cols] = -np.inf
    kc, comp, err = run_gpu_ex(p)
    assert err == 0
    rep = check_against_oracle_ex(p, kc, comp)
    assert rep["stored"] > 0
