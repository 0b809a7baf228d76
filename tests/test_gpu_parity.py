"""CUDA path vs the CPU oracle, element by element, through the C-ABI.

Two levels (the compressed fp32 vector is only defined up to rounding order):
  (i)  the oracle's epilogue applied to the GPU's own comp32 reproduces every k_cache byte
       (FP8 codes, UE8M0 scales, bf16 rope values, untouched bytes) exactly;
  (ii) the GPU's comp32 is within 1e-6 + 1e-5*|x| of the oracle's (binary64 softmax), and every
       byte that differs from the oracle's own output sits in a window whose comp32 differs.
"""
import numpy as np
import pytest

import oracle
from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import check_against_oracle, run_gpu, to_device, written_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_v4_sparse_c128_gb300 import build, binding
    build.build()
    binding.load()


@pytest.mark.parametrize("name", ["tiny", "decode", "mixed", "varlen16k", "varlen"])
def test_workload_parity(name):
    p = inputs.make_problem(name)
    kc, comp, err = run_gpu(p)
    assert err == 0
    rep = check_against_oracle(p, kc, comp, threads=16)
    print(name, rep)
    if name == "tiny":
        assert rep["stored"] == 4
    if name == "mixed":  # ~1/128 of 4096 at a window end, minus the padded ones
        assert 10 <= rep["stored"] <= 60


@pytest.mark.parametrize("T", [1, 2, 3, 5, 19, 20, 38, 39, 64, 76, 77, 127, 151, 152, 153, 200, 256, 300, 600, 1000, 1216, 1217, 2000])
def test_sweep_sizes(T):
    """All-boundary tokens: every launch mode (cluster split S = 8, 4, 2, 1 for T x S <= #SM,
    then the planned persistent path, whose windows are split into 8, 4, 2 or 1 parts merged
    through the workspace) and the edges between them, past the SM count (ragged last wave)."""
    p = inputs.make_problem("sweep", tokens=T)
    kc, comp, err = run_gpu(p)
    assert err == 0
    rep = check_against_oracle(p, kc, comp, threads=16)
    assert rep["stored"] == T


@pytest.mark.parametrize("seed", range(6))
def test_random_problems(seed):
    """Padded tokens, negative positions, missing kv slots, aliased blocks, kv block sizes 1..64."""
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([1, 2, 3, 16, 64]))
    p = inputs.random_problem(1000 + seed, num_tokens=int(rng.integers(50, 700)), num_reqs=7, max_blocks=96,
                              num_blocks=int(rng.integers(20, 200)), kv_block_size=bs,
                              active_frac=float(rng.uniform(0.1, 0.9)))
    kc, comp, err = run_gpu(p)
    assert err == 0
    check_against_oracle(p, kc, comp, threads=16)


def test_empty_and_all_inactive():
    import torch
    p = inputs.random_problem(77, num_tokens=300, num_reqs=3, max_blocks=64, num_blocks=50, kv_block_size=2,
                              active_frac=0.0)
    p.positions[:] = 5  # never a window end
    kc, comp, err = run_gpu(p)
    assert err == 0 and np.array_equal(kc, p.k_cache) and written_rows(comp).size == 0
    # T == 0 is a no-op that returns OK
    q = inputs.random_problem(78, num_tokens=0, num_reqs=1, max_blocks=8, num_blocks=4, kv_block_size=2)
    kc0, _, err0 = run_gpu(q, comp=False)
    assert err0 == 0 and np.array_equal(kc0, q.k_cache)
    assert torch.cuda.is_available()


def _strided(dev, key, pad_shape, sl):
    import torch
    src = dev[key]
    big = torch.zeros(pad_shape, dtype=src.dtype, device=src.device)
    view = big[sl]
    view.copy_(src)
    dev[key] = view
    return view


def take_tokens(p, n):
    """The first n tokens of a problem (same caches)."""
    return inputs.Problem(p.name + f"[:{n}]", p.token_to_req[:n].copy(), p.positions[:n].copy(),
                          p.slot_mapping[:n].copy(), p.block_table, p.state, p.rms_w, p.eps, p.cos_sin, p.k_cache,
                          p.kv_slot_mapping[:n].copy(), p.kv_block_size)


@pytest.mark.parametrize("name,n", [("decode", 128), ("decode", 12), ("mixed", 4096)])
def test_padded_strides(name, n):
    """Non-contiguous state rows (per-row copies), padded blocks, padded block-table rows, padded
    cos/sin rows, padded k_cache blocks with wider records; direct and planned launch modes."""
    import torch
    p = take_tokens(inputs.make_problem(name), n)
    dev = to_device(p)
    NB = p.state.shape[0]
    _strided(dev, "state", (NB, 8, 1152 + 64), (slice(None), slice(None), slice(0, 1024)))
    assert dev["state"].stride(1) == 1216 and dev["state"].stride(0) == 8 * 1216
    R, MB = p.block_table.shape
    _strided(dev, "block_table", (R, MB + 5), (slice(None), slice(0, MB)))
    MP = p.cos_sin.shape[0]
    _strided(dev, "cos_sin", (MP, 68), (slice(None), slice(0, 64)))
    NKB, bs, W = p.k_cache.shape
    big = torch.randint(0, 256, (NKB, bs * 600 + 16), dtype=torch.uint8, device="cuda")
    kview = big[:, :bs * 600].view(NKB, bs, 600)
    # place the original records at the same logical offsets: block layout is flat bytes
    kview.view(NKB, -1)[:, :bs * 584].copy_(dev["k_cache"].view(NKB, -1))
    before = big.clone()
    dev["k_cache"] = kview
    kc, comp, err = run_gpu(p, dev=dev)
    assert err == 0
    rows = written_rows(comp)
    # expected: the oracle epilogue on the GPU's comp32 (compact layout), transplanted into the
    # padded buffer: a block is a flat byte range, so the record offsets do not depend on W
    from gpu_util import replay_expected
    exp = before.cpu().numpy()
    exp[:, :bs * 584] = replay_expected(p, comp, rows).reshape(NKB, -1)
    assert np.array_equal(big.cpu().numpy(), exp)
    rep = check_against_oracle(p, replay_expected(p, comp, rows), comp)
    assert rep["stored"] == rows.size > 0


def test_paging_invariance_gpu():
    p = inputs.make_problem("decode")
    kc_a, comp_a, _ = run_gpu(p)
    rng = np.random.default_rng(5)
    perm = rng.permutation(p.state.shape[0])
    st = np.empty_like(p.state)
    st[perm] = p.state
    p.state = st
    p.block_table = perm[p.block_table].astype(np.int32)
    kc_b, comp_b, _ = run_gpu(p)
    assert np.array_equal(kc_a, kc_b)
    assert np.array_equal(comp_a.view(np.uint32), comp_b.view(np.uint32))


@pytest.mark.parametrize("which", ["decode", "decode16", "sweep300"])
def test_bad_indices_are_reported_and_skipped(which):
    """Out-of-range request / block-table column / block id / cos row / kv slot: the token writes
    nothing, the matching device error bit is set, every other token is stored normally
    (direct S = 1, cluster-split S = 8 and planned launch modes)."""
    if which == "decode":
        p = inputs.make_problem("decode")
    elif which == "decode16":
        p = take_tokens(inputs.make_problem("decode"), 16)
    else:
        p = inputs.make_problem("sweep", tokens=300)
    bt_cols = p.block_table.shape[1]
    p.token_to_req[3] = p.block_table.shape[0]          # BAD_REQ
    p.positions[5] = bt_cols * 8 + 127                  # BAD_BT_COL (a window end past the table)
    first = (int(p.positions[7]) - 127) // 8
    p.block_table[int(p.token_to_req[7]), first + 9] = p.state.shape[0]  # BAD_BLOCK
    p.kv_slot_mapping[9] = p.k_cache.shape[0] * p.kv_block_size           # BAD_KV_SLOT
    p.cos_sin = p.cos_sin[:4096]                         # BAD_COS_ROW for windows starting >= 4096
    kc, comp, err = run_gpu(p)
    ref = p.k_cache.copy()
    err_ref = oracle.forward(p, k_cache=ref)
    assert err == err_ref
    assert err & (1 | 2 | 4 | 8 | 16) == (1 | 2 | 4 | 8 | 16)
    rep = check_against_oracle(p, kc, comp)      # same stored set, same bytes
    assert not {3, 5, 7, 9} & set(written_rows(comp).tolist())
    assert 0 < rep["stored"] < p.num_tokens - 4


@pytest.mark.parametrize("n", [128, 16])
def test_one_hot_epilogue_edges(n):
    """Scores 0 on one row and -1000 elsewhere make comp32 equal that row's kv exactly on both
    sides, so crafted comp vectors reach the epilogue: huge dynamic range (exact-variance slow
    path), subnormals, zeros, exact bf16/e4m3 ties, overflowing variance. n = 16 runs the
    cluster-split launch, whose partial softmax states are merged across 8 CTAs."""
    rng = np.random.default_rng(9)
    p = take_tokens(inputs.make_problem("decode"), n)
    T = p.num_tokens
    pick = rng.integers(0, 128, size=(T, 512))
    vals = np.zeros((T, 512), np.float32)
    for t in range(T):
        kind = t % 8
        if kind == 0:
            v = rng.standard_normal(512) * 2.0 ** rng.integers(-60, 40, 512)        # > 2^32 spread
        elif kind == 1:
            v = rng.standard_normal(512) * 1e-40                                    # subnormal
        elif kind == 2:
            v = np.zeros(512)
        elif kind == 3:
            v = np.where(rng.random(512) < 0.5, 0.0, rng.standard_normal(512))
        elif kind == 4:
            v = (1 + np.arange(512) % 7 / 64.0) * rng.choice([-1, 1], 512)           # tie-prone
        elif kind == 5:
            v = rng.standard_normal(512) * 1e25                                     # var overflows
        elif kind == 6:
            v = rng.standard_normal(512) * 1e-20
        else:
            v = rng.standard_normal(512)
        vals[t] = v.astype(np.float32)
    # every score row of the window -> -1000 except the picked one; write the picked kv values
    for t in range(T):
        r = int(p.token_to_req[t])
        start = int(p.positions[t]) - 127
        q = start + np.arange(128)
        blocks = p.block_table[r, q // 8]
        sc = np.full((128, 512), -1000.0, np.float32)   # exp(-1000) is 0 in binary64 too
        sc[pick[t], np.arange(512)] = 0.0
        p.state[blocks, q % 8, 512:] = sc
        p.state[blocks[pick[t]], (q % 8)[pick[t]], np.arange(512)] = vals[t]
    kc, comp, err = run_gpu(p)
    assert err == 0
    assert np.array_equal(comp.view(np.uint32), vals.view(np.uint32))
    rep = check_against_oracle(p, kc, comp, threads=16)
    assert rep["e2e_bytes_differ"] == 0


def test_full_size_sweep_sampled():
    """token_num = 16374 (8.6 GB of state drawn on the device), the launch the benchmark times:
    every window's bytes checked by epilogue replay, a sample of 768 windows against the oracle's
    own softmax."""
    import torch
    p = inputs.make_problem("sweep", tokens=16374, state_device="cuda")
    dev = to_device(p)
    kc, comp, err = run_gpu(p, dev=dev)
    assert err == 0
    rows = written_rows(comp)
    assert rows.size == 16374
    from gpu_util import replay_expected, comp_close
    assert np.array_equal(replay_expected(p, comp, rows), kc)
    rng = np.random.default_rng(3)
    sample = np.unique(np.concatenate([[0, 16373], rng.choice(16374, 766, replace=False)]))
    # compact host problem holding only the sampled windows' blocks
    first = (p.positions[sample] - 127) // 8
    blk = np.stack([p.block_table[sample[i], first[i]:first[i] + 16] for i in range(sample.size)])
    st = dev["state"].index_select(0, torch.from_numpy(blk.reshape(-1).astype(np.int64)).cuda()).cpu().numpy()
    sub = inputs.Problem("sample", np.arange(sample.size, dtype=np.int32), p.positions[sample].copy(),
                         p.slot_mapping[sample].copy(), np.zeros((sample.size, 1024), np.int32), st, p.rms_w,
                         p.eps, p.cos_sin, p.k_cache, p.kv_slot_mapping[sample].copy(), p.kv_block_size)
    for i in range(sample.size):
        sub.block_table[i, first[i]:first[i] + 16] = np.arange(16 * i, 16 * i + 16)
    comp_ref = np.zeros((sample.size, 512), np.float32)
    oracle.forward(sub, k_cache=sub.k_cache.copy(), comp_out=comp_ref, threads=16)
    ok, max_abs, worst = comp_close(comp[sample], comp_ref)
    print("sweep16374 sample: max abs", max_abs, "worst/tol", worst)
    assert ok


def test_streams_graphs_and_timer():
    """Two streams (separate workspaces), CUDA-graph capture after reserve_workspace, and the
    kernel timer counting launches."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    p = inputs.make_problem("decode")
    ref = oracle.forward_k_cache(p)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    d1, d2 = to_device(p), to_device(p)
    torch.cuda.synchronize()
    for s, d in ((s1, d1), (s2, d2)):
        with torch.cuda.stream(s):
            binding.compress_norm_rope_store(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                             d["state"], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
                                             d["kv_slot_mapping"], p.kv_block_size)
    torch.cuda.synchronize()
    got1, got2 = d1["k_cache"].cpu().numpy(), d2["k_cache"].cpu().numpy()
    assert np.array_equal(got1, got2)
    kc_gpu, comp, _ = run_gpu(p)
    assert np.array_equal(kc_gpu, got1)
    # graph capture
    d3 = to_device(p)
    s3 = torch.cuda.Stream()
    with torch.cuda.stream(s3):
        binding.reserve_workspace(p.num_tokens)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s3):
        binding.compress_norm_rope_store(d3["token_to_req"], d3["positions"], d3["slot_mapping"], d3["block_table"],
                                         d3["state"], d3["rms_w"], p.eps, d3["cos_sin"], d3["k_cache"],
                                         d3["kv_slot_mapping"], p.kv_block_size)
    d3["k_cache"].copy_(torch.from_numpy(p.k_cache).cuda())
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(d3["k_cache"].cpu().numpy(), got1)
    # timer
    with binding.KernelTimer() as tm:
        for _ in range(3):
            binding.compress_norm_rope_store(d1["token_to_req"], d1["positions"], d1["slot_mapping"],
                                             d1["block_table"], d1["state"], d1["rms_w"], p.eps, d1["cos_sin"],
                                             d1["k_cache"], d1["kv_slot_mapping"], p.kv_block_size)
    assert tm.launches == 3 and tm.total_ms > 0
    assert ref is not None


@pytest.mark.parametrize("tokens", [300, 2000])  # one CTA per token; planning pass + PDL
def test_graph_capture_c128_paths(tokens):
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    p = inputs.make_problem("sweep", tokens=tokens)
    kc_eager, _, err = run_gpu(p, comp=False)
    assert err == 0
    d = to_device(p)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        binding.reserve_workspace(p.num_tokens)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.compress_norm_rope_store(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                         d["state"], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
                                         d["kv_slot_mapping"], p.kv_block_size)
    for _ in range(2):
        d["k_cache"].copy_(torch.from_numpy(p.k_cache).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(d["k_cache"].cpu().numpy(), kc_eager)
    assert binding.device_errors(s, clear=True) == 0


def test_prepared_call_matches_function_call():
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    p = inputs.make_problem("mixed")
    kc_ref, comp_ref, _ = run_gpu(p)
    d = to_device(p)
    comp = torch.zeros((p.num_tokens, 512), dtype=torch.float32, device="cuda")
    call = binding.PreparedCall(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"], d["state"],
                                d["rms_w"], p.eps, d["cos_sin"], d["k_cache"], d["kv_slot_mapping"], p.kv_block_size,
                                comp_out=comp)
    call()
    call()  # idempotent: same inputs, same bytes
    torch.cuda.synchronize()
    assert np.array_equal(d["k_cache"].cpu().numpy(), kc_ref)
    rows = written_rows(comp_ref)
    assert np.array_equal(comp.cpu().numpy()[rows].view(np.uint32), comp_ref[rows].view(np.uint32))


def test_host_validation_on_gpu():
    """Layout errors are rejected before anything is launched."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    p = inputs.make_problem("tiny")
    d = to_device(p)
    args = lambda **kw: [kw.get(k, d[k]) for k in ("token_to_req", "positions", "slot_mapping", "block_table",
                                                     "state")] + [d["rms_w"], p.eps, d["cos_sin"],
                                                                  kw.get("k_cache", d["k_cache"]),
                                                                  d["kv_slot_mapping"], kw.get("bs", p.kv_block_size)]
    assert binding.call_status(*args()) == 0
    assert binding.call_status(*args(bs=4)) == 7
    assert binding.call_status(*args(positions=d["positions"].int())) == 2
    assert binding.call_status(*args(state=d["state"][:, :4])) == 6
    assert binding.call_status(*args(token_to_req=d["token_to_req"][:3])) == 3
    bad = torch.zeros(p.state.shape[0], 8, 1024 + 1, device="cuda")[:, :, 1:]
    assert binding.call_status(*args(state=bad)) == 5
