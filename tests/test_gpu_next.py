"""CUDA path vs the CPU oracle for the other configurations of the pages' fused kernels, through
compress_norm_rope_store_ex: C4 overlapping windows with the sparse-attention cache (head 512),
and the head-128 indexer with an FP8 (fp32 scale) or MXFP4 (UE8M0) cache at compress ratios 4
(overlap) and 128. Same two-level parity as the C128 tests."""
import numpy as np
import pytest

import oracle
from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import (check_against_oracle_ex, run_gpu, run_gpu_ex, to_device, written_rows)

pytestmark = pytest.mark.gpu

NEXT = ["c4_sparse", "idx_c4_fp8", "idx_c4_mxfp4", "idx_c128_fp8", "idx_c128_mxfp4"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_v4_sparse_c128_gb300 import build, binding
    build.build()
    binding.load()


@pytest.mark.parametrize("name", NEXT)
def test_next_workload_parity(name):
    p = inputs.make_next_problem(name)
    kc, comp, err = run_gpu_ex(p)
    assert err == 0
    rep = check_against_oracle_ex(p, kc, comp, threads=16)
    print(name, rep)
    assert rep["stored"] > 100


@pytest.mark.parametrize("block", [1, 4, 16, 32])
@pytest.mark.parametrize("fmt,head", [(0, 512), (2, 128)])
def test_other_state_block_sizes(block, fmt, head):
    p = inputs.prefill_problem("blk", 11 + block, 6, 5, 300, head, 4, 1, fmt, state_block=block, kv_block_size=16,
                               decode_tail=5)
    kc, comp, err = run_gpu_ex(p)
    assert err == 0
    check_against_oracle_ex(p, kc, comp, threads=16)


@pytest.mark.parametrize("block", [1, 4, 8, 16, 64])
@pytest.mark.parametrize("fmt,ratio,overlap", [(1, 16, 1), (2, 128, 0), (1, 8, 1)])
def test_indexer_long_windows_block_sizes(block, fmt, ratio, overlap):
    """Head-128 windows longer than 8 rows: state blocks that are multiples of 8 rows take the
    tiled-load ring kernel, the others the gather kernel; both against the oracle."""
    p = inputs.prefill_problem("ixblk", 31 + block, 5, 5, 40 * ratio, 128, ratio, overlap, fmt, state_block=block,
                               kv_block_size=16, decode_tail=6)
    kc, comp, err = run_gpu_ex(p)
    assert err == 0
    rep = check_against_oracle_ex(p, kc, comp, threads=16)
    assert rep["stored"] > 10


def test_c128_config_through_ex_is_the_c128_call():
    for name in ("decode", "mixed"):
        p = inputs.make_problem(name)
        a, ca, _ = run_gpu(p)
        b, cb, _ = run_gpu_ex(p)
        assert np.array_equal(a, b)
        rows = written_rows(ca)
        assert np.array_equal(ca[rows].view(np.uint32), cb[rows].view(np.uint32))


@pytest.mark.parametrize("sblk", [16, 24, 64, 128, 256, 12, 20])
@pytest.mark.parametrize("shape", ["direct", "per_token", "planned"])
def test_c128_config_with_other_block_sizes(sblk, shape):
    """C128 sizes with state blocks other than 8 rows: multiples of 8 take the C128 kernels (a
    window's 8-row chunks sit at row q0 % sblk of block q0 / sblk), others the generic kernel; each
    launch mode of the C128 kernels (cluster split up to #SM tokens, one CTA per token up to 8 per SM,
    then the planning pass), checked against the oracle."""
    reqs, lo, hi = {"direct": (1, 128, 128), "per_token": (1, 600, 600), "planned": (3, 128, 3000)}[shape]
    p = inputs.prefill_problem(f"c128b{sblk}", 5 + sblk, reqs, lo, hi, 512, 128, 0, 0, state_block=sblk,
                               decode_tail=20)
    kc, comp, err = run_gpu_ex(p)
    assert err == 0
    rep = check_against_oracle_ex(p, kc, comp, threads=16)
    assert rep["stored"] > 0


def test_c128_config_other_block_size_bad_indices():
    """16-row state blocks on the C128 kernels: an out-of-range block id (BAD_BLOCK) and a window
    end past the block table (BAD_BT_COL) are reported and skipped like with 8-row blocks."""
    p = inputs.prefill_problem("c128b16bad", 9, 2, 1000, 2000, 512, 128, 0, 0, state_block=16, decode_tail=40)
    act = np.nonzero((p.positions + 1) % 128 == 0)[0]
    t1, t2 = int(act[3]), int(act[-2])
    r1 = int(p.token_to_req[t1])
    p.block_table[r1, (int(p.positions[t1]) - 127) // 16 + 3] = p.state.shape[0]   # BAD_BLOCK
    p.positions[t2] = p.block_table.shape[1] * 16 + 127                             # BAD_BT_COL
    kc, comp, err = run_gpu_ex(p)
    ref = p.k_cache.copy()
    assert err == oracle.forward_ex(p, k_cache=ref) and err & (2 | 4) == (2 | 4)
    check_against_oracle_ex(p, kc, comp, threads=16)


@pytest.mark.parametrize("name", ["idx_c4_fp8", "c4_sparse", "idx_c128_mxfp4"])
def test_bad_indices_generic_path(name):
    p = inputs.make_next_problem(name)
    act = [t for t in range(p.num_tokens) if p.kv_slot_mapping[t] >= 0 and p.positions[t] >= 7]
    t_req, t_blk, t_kv, t_bt = act[3], act[10], act[20], act[30]
    p.token_to_req[t_req] = p.block_table.shape[0]
    r = int(p.token_to_req[t_blk])
    q = int(p.positions[t_blk]) - 2
    p.block_table[r, q // p.state.shape[1]] = p.state.shape[0]
    p.kv_slot_mapping[t_kv] = p.k_cache.shape[0] * p.kv_block_size
    p.positions[t_bt] = p.block_table.shape[1] * p.state.shape[1] + p.ratio - 1  # a window end past the table
    kc, comp, err = run_gpu_ex(p)
    ref = p.k_cache.copy()
    err_ref = oracle.forward_ex(p, k_cache=ref)
    assert err == err_ref and err & (1 | 2 | 4 | 16) == (1 | 2 | 4 | 16)
    rep = check_against_oracle_ex(p, kc, comp)
    assert not {t_req, t_blk, t_kv, t_bt} & set(written_rows(comp).tolist())
    assert rep["stored"] > 0


@pytest.mark.parametrize("fmt,head,ratio,overlap", [(1, 128, 4, 1), (2, 128, 4, 1), (0, 512, 4, 1),
                                                   (1, 128, 128, 0), (2, 128, 128, 0), (2, 128, 16, 1)])
def test_one_hot_epilogue_edges_generic(fmt, head, ratio, overlap):
    """One-hot scores (0 on one valid row, -1000 elsewhere) make comp32 equal crafted kv values on
    both sides: wide dynamic range (slow exact variance), subnormals, zeros, E2M1/e4m3 ties,
    tiny blocks (MXFP4 scale near 2^-127), an overflowing variance. Windows of up to 8 rows run
    the small-window kernel, longer head-128 windows the tiled-load ring kernel, longer head-512
    windows the gather kernel."""
    nrows = (1 + overlap) * ratio
    p = inputs.prefill_problem("onehot", 21, 4, max(8, ratio), max(64, 4 * ratio), head, ratio, overlap, fmt,
                               decode_tail=8)
    rng = np.random.default_rng(fmt)
    sw = p.state_width
    p.state[..., sw:] = -1000.0
    rows_tok = [t for t in range(p.num_tokens) if p.kv_slot_mapping[t] >= 0]
    want = {}
    for n, t in enumerate(rows_tok):
        kind = n % 8
        if kind == 0:
            v = rng.standard_normal(head) * 2.0 ** rng.integers(-60, 40, head)
        elif kind == 1:
            v = rng.standard_normal(head) * 1e-40
        elif kind == 2:
            v = np.zeros(head)
        elif kind == 3:
            v = rng.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -2.5], head) * 2.0 ** rng.integers(-3, 3)
        elif kind == 4:
            v = rng.standard_normal(head) * 1e25
        elif kind == 5:
            v = rng.standard_normal(head) * 1e-30
        else:
            v = rng.standard_normal(head)
        pos, r = int(p.positions[t]), int(p.token_to_req[t])
        valid = [i for i in range(nrows) if pos - nrows + 1 + i >= 0]
        pick = rng.choice(valid, head)
        for c in range(head):
            q = pos - nrows + 1 + pick[c]
            ho = head if pick[c] >= ratio else 0
            b, o = p.block_table[r, q // 8], q % 8
            p.state[b, o, sw + ho + c] = 0.0
            p.state[b, o, ho + c] = np.float32(v[c])
        want[t] = v.astype(np.float32)
    kc, comp, err = run_gpu_ex(p)
    assert err == 0
    for t, v in want.items():
        assert np.array_equal(comp[t].view(np.uint32), v.view(np.uint32)), t
    rep = check_against_oracle_ex(p, kc, comp)
    assert rep["e2e_bytes_differ"] == 0


@pytest.mark.parametrize("name", ["idx_c4_mxfp4", "idx_c128_fp8", "c4_sparse", "idx_c4_fp8"])
def test_padded_strides_generic(name):
    """Padded state rows, padded block-table rows, cos/sin rows of 66 floats (rows not 16-byte
    aligned) and k_cache blocks wider than their records: the ring kernels address everything
    through the strides."""
    import torch
    from gpu_util import FORMAT_BYTES, replay_expected_ex
    p = inputs.make_next_problem(name)
    dev = to_device(p)
    NB, BS, RW = p.state.shape
    big = torch.zeros((NB, BS, RW + 36), dtype=torch.float32, device="cuda")
    big[:, :, :RW].copy_(dev["state"])
    dev["state"] = big[:, :, :RW]
    R, MB = p.block_table.shape
    bt = torch.zeros((R, MB + 5), dtype=torch.int32, device="cuda")
    bt[:, :MB].copy_(dev["block_table"])
    dev["block_table"] = bt[:, :MB]
    MP = p.cos_sin.shape[0]
    cs = torch.zeros((MP, 66), dtype=torch.float32, device="cuda")
    cs[:, :64].copy_(dev["cos_sin"])
    dev["cos_sin"] = cs[:, :64]
    tb, sb = FORMAT_BYTES[p.fmt]
    NKB, bs, W = p.k_cache.shape
    Wp = tb + sb + 16
    kbig = torch.randint(0, 256, (NKB, bs * Wp + 16), dtype=torch.uint8, device="cuda")
    kview = kbig[:, :bs * Wp].view(NKB, bs, Wp)
    kview.view(NKB, -1)[:, :bs * (tb + sb)].copy_(dev["k_cache"].view(NKB, -1))
    before = kbig.cpu().numpy()
    dev["k_cache"] = kview
    kc, comp, err = run_gpu_ex(p, dev=dev)
    assert err == 0
    rows = written_rows(comp)
    exp = before.copy()
    exp[:, :bs * (tb + sb)] = replay_expected_ex(p, comp, rows).reshape(NKB, -1)
    assert np.array_equal(kbig.cpu().numpy(), exp)
    rep = check_against_oracle_ex(p, replay_expected_ex(p, comp, rows), comp)
    assert rep["stored"] == rows.size > 0


@pytest.mark.parametrize("name", ["c4_sparse", "idx_c4_fp8", "idx_c128_mxfp4"])
def test_graph_capture_generic(name):
    """The ring kernels (tensor map encoded on the host at launch) captured in a CUDA graph and
    replayed give the eager call's bytes."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    p = inputs.make_next_problem(name)
    kc_eager, _, err = run_gpu_ex(p, comp=False)
    assert err == 0
    d = to_device(p)
    cfg = binding.config(p.head, p.ratio, p.overlap, p.state_width, p.fmt)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        binding.reserve_workspace(p.num_tokens)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.compress_norm_rope_store_ex(cfg, d["token_to_req"], d["positions"], d["slot_mapping"],
                                            d["block_table"], d["state"], d["rms_w"], p.eps, d["cos_sin"],
                                            d["k_cache"], d["kv_slot_mapping"], p.kv_block_size)
    for _ in range(2):
        d["k_cache"].copy_(torch.from_numpy(p.k_cache).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(d["k_cache"].cpu().numpy(), kc_eager)
    assert binding.device_errors(s, clear=True) == 0


@pytest.mark.parametrize("name", NEXT)
def test_next_bench_size_sampled(name):
    """Each configuration at the size bench.py times (about a quarter million tokens, state drawn
    on the device, larger than L2): the stored set equals the activity predicate, every stored
    slot equals the oracle epilogue replayed on the GPU's comp32, and 256 sampled windows' comp32
    match the oracle within 1e-6 + 1e-5|x|."""
    import dataclasses
    import bench
    from gpu_util import comp_close, replay_expected_ex, NAN_BITS
    p = inputs.make_next_problem(name, state_device="cuda", scale=bench.NEXT_SCALES[name])
    kc, comp, err = run_gpu_ex(p, dev=to_device(p))
    assert err == 0
    ph = dataclasses.replace(p, state=p.state.cpu().numpy())
    rows = written_rows(comp)
    active = np.nonzero((p.slot_mapping >= 0) & (p.positions >= 0) & ((p.positions + 1) % p.ratio == 0) &
                        (p.kv_slot_mapping >= 0))[0]
    assert np.array_equal(rows, active)
    assert np.array_equal(replay_expected_ex(ph, comp, rows), kc)
    sample = np.sort(np.random.default_rng(5).choice(rows, size=min(256, rows.size), replace=False))
    comp_ref = np.zeros((p.num_tokens, p.head), np.float32)
    comp_ref.view(np.uint32)[:] = NAN_BITS
    oracle.forward_ex(ph, k_cache=ph.k_cache.copy(), tokens=sample, comp_out=comp_ref, threads=16)
    ok, max_abs, worst = comp_close(comp[sample], comp_ref[sample])
    assert ok, (max_abs, worst)
