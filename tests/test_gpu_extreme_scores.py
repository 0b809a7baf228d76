"""Extreme scores through the whole path, against the oracle (two-level parity):
- -inf scores on random rows of random columns (never a whole column): those rows get weight 0,
  as in a masked softmax;
- scores scaled by 1e4: nearly one-hot weights, where exp(s - max) underflows for all but the top
  rows and nothing may overflow;
- scores offset by +1e4 or -1e4 per state block: large magnitudes, where within a window the
  blocks with the lower offset get weights that underflow to 0.
Each on every C128 call path (cluster split, token striding, planning pass)."""
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
