"""Pins for the oracle's generalised gather: any compress ratio, with or without overlap, any
state block size and any state width (c128o_forward_ex).

The gather is the one the API page prints in each fused kernel of
vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache, section "Gather state cache
entries": a window ending at position p covers the (1 + OVERLAP) * COMPRESS_RATIO positions
p - (1 + OVERLAP) * COMPRESS_RATIO + 1 .. p; position q is row q % block_size of block
block_table[req, q // block_size]; rows at negative positions are masked out of the softmax
(score -inf, kv 0); the newer COMPRESS_RATIO rows of an overlapping window read kv and score at
+HEAD_SIZE (head_offset); score columns follow the STATE_WIDTH kv columns of a row. The RoPE row
is (p // COMPRESS_RATIO) * COMPRESS_RATIO (compressed_pos), and the slot record sits at
kv_slot // kv_cache_block_size, kv_slot % kv_cache_block_size of the k_cache.

Three independent checks:
* identity-coded gathers: every kv value names its physical (block, row, column), one score per
  column is 0 on a chosen window row, the window's other rows score -1000 and every row outside
  the window scores +500, so a window that is too long, too short or shifted, a wrong row or
  block, a wrong half or a wrong column gives a different number;
* re-blocking invariance: the same logical rows laid out with state blocks of 1..64 rows give
  identical k_cache bytes and compressed vectors;
* brute force: a float64 numpy re-derivation of the column softmax and weighted sum, written
  from the definition above, on random data.
"""
import math

import numpy as np
import pytest

import oracle
from deepseek_v4_sparse_c128_gb300 import inputs

# token / scale bytes of a k_cache slot per cache format (sparse FP8 + bf16 rope; indexer FP8 +
# fp32 scale; indexer MXFP4 + 4 UE8M0 bytes), as the cache-layout docstrings on the API page give
SLOT = {0: (576, 8), 1: (128, 4), 2: (64, 4)}


def _paged_problem(rng, lens, head, ratio, overlap, fmt, sb, sw=None, kv_bs=4, logical=None):
    """Requests with every position 0..len-1 present. Every block-table entry is a distinct block
    (no aliasing), with one spare block past each request's last position. ``logical`` (a list of
    per-request [rows, 2*sw] arrays) fixes the row contents; otherwise they are drawn."""
    sw = sw or head * (1 + overlap)
    lens = [int(n) for n in lens]
    R = len(lens)
    MB = max(-(-(n + 1) // sb) for n in lens) + 1
    NB = R * MB
    bt = rng.permutation(NB).reshape(R, MB).astype(np.int32)
    state = rng.standard_normal((NB, sb, 2 * sw)).astype(np.float32)
    state[..., sw:] *= np.float32(2.0)
    if logical is not None:
        for r in range(R):
            for q in range(lens[r]):
                state[bt[r, q // sb], q % sb] = logical[r][q]
    req = np.concatenate([np.full(n, r, np.int32) for r, n in enumerate(lens)])
    pos = np.concatenate([np.arange(n, dtype=np.int64) for n in lens])
    slot = (bt[req, pos // sb].astype(np.int64) * sb + pos % sb)
    T = pos.shape[0]
    NKB = -(-T // kv_bs)
    kv_slot = rng.permutation(NKB * kv_bs)[:T].astype(np.int64)
    tok, sc = SLOT[fmt]
    k_cache = rng.integers(0, 256, size=(NKB, kv_bs, tok + sc), dtype=np.uint8)
    cos_sin = rng.uniform(-1, 1, size=(max(lens) + 1, 64)).astype(np.float32)
    rms_w = (1.0 + 0.1 * rng.standard_normal(head)).astype(np.float32)
    return inputs.Problem("gather-pin", req, pos, slot, bt, state, rms_w, 1e-6, cos_sin, k_cache, kv_slot, kv_bs,
                          head=head, ratio=ratio, overlap=overlap, state_width=sw, fmt=fmt)


def _window_rows(p, ratio, overlap):
    """(window row index i, position q) for each row of the window ending at p; rows i >= ratio
    are the newer half."""
    n = (1 + overlap) * ratio
    return [(i, p - n + 1 + i) for i in range(n)]


def _epilogue(fmt, comp, pr, p):
    cs = pr.cos_sin[(p // pr.ratio) * pr.ratio]
    if fmt == 0:
        return oracle.epilogue(comp, pr.rms_w, pr.eps, cs)
    return oracle.epilogue_indexer(fmt, comp, pr.rms_w, pr.eps, cs)


def _slot_bytes(k_cache, fmt, bs, kvs):
    """(token bytes, scale bytes) of slot kvs, at the addresses the API page's store uses."""
    tok, sc = SLOT[fmt]
    blk = k_cache[kvs // bs].reshape(-1)
    off = kvs % bs
    return blk[off * tok:(off + 1) * tok], blk[bs * tok + off * sc:bs * tok + (off + 1) * sc]


def _active(pr):
    p = pr.positions
    return np.nonzero((pr.slot_mapping >= 0) & (p >= 0) & ((p + 1) % pr.ratio == 0) & (pr.kv_slot_mapping >= 0))[0]


# (head, ratio, overlap, format, state block, state width or None for (1 + overlap) * head)
IDENTITY_CASES = [
    (128, 1, 0, 1, 1, None), (128, 1, 1, 2, 3, None), (128, 2, 0, 2, 1, None), (128, 2, 1, 1, 2, None),
    (128, 8, 0, 1, 8, None), (128, 8, 1, 2, 4, None), (128, 16, 0, 1, 16, 192), (128, 16, 1, 1, 8, None),
    (128, 16, 1, 2, 5, 288), (128, 64, 0, 2, 64, None), (128, 64, 1, 1, 16, None), (128, 128, 1, 1, 8, None),
    (128, 256, 0, 2, 32, None), (512, 4, 1, 0, 2, None), (512, 16, 1, 0, 16, None), (512, 128, 0, 0, 16, None),
    (512, 64, 0, 0, 1, None),
]


@pytest.mark.parametrize("head,ratio,overlap,fmt,sb,sw", IDENTITY_CASES)
def test_identity_coded_gather(head, ratio, overlap, fmt, sb, sw):
    """Each column's one-hot score picks one window row; the compressed value must be the kv code
    of exactly that (block, row, half, column), and the record must land in the token's slot."""
    rng = np.random.default_rng([head, ratio, overlap, fmt, sb])
    n = (1 + overlap) * ratio
    lens = [n + int(rng.integers(0, n + 3)), n + int(rng.integers(0, 2 * n)), 2 * n + 1]
    pr = _paged_problem(rng, lens, head, ratio, overlap, fmt, sb, sw)
    sw = pr.state_width
    NB = pr.state.shape[0]
    assert NB * sb * 2048 < 2 ** 24                          # codes stay exact integers in fp32
    code = (np.arange(NB)[:, None] * sb + np.arange(sb)[None, :]).astype(np.int64) * 2048
    pr.state[..., :sw] = (code[..., None] + np.arange(sw)[None, None, :]).astype(np.float32)
    base_state = pr.state.copy()
    act = _active(pr)
    req_first = {}
    for t in act:
        req_first.setdefault(int(pr.token_to_req[t]), int(t))
    chosen = sorted(set(req_first.values()) | {int(act[-1]), int(act[len(act) // 2])})
    for t in chosen:
        p, r = int(pr.positions[t]), int(pr.token_to_req[t])
        st = base_state.copy()
        st[..., sw:] = 500.0                                   # every row outside the window
        valid = []
        for i, q in _window_rows(p, ratio, overlap):
            if q < 0:
                continue
            ho = head if i >= ratio else 0
            st[bt_blk(pr, r, q, sb), q % sb, sw + ho:sw + ho + head] = -1000.0
            valid.append(i)
        if overlap and p == ratio - 1:
            assert len(valid) == ratio                       # the older half is all masked
        pick = rng.choice(valid, head)
        pick[: min(head, 2)] = [valid[0], valid[-1]]         # the oldest and the newest row
        q = p - n + 1 + pick
        ho = np.where(pick >= ratio, head, 0)
        blk = pr.block_table[r, q // sb].astype(np.int64)
        cols = np.arange(head)
        st[blk, q % sb, sw + ho + cols] = 0.0
        sub = inputs.Problem("x", pr.token_to_req, pr.positions, pr.slot_mapping, pr.block_table, st, pr.rms_w,
                             pr.eps, pr.cos_sin, pr.k_cache, pr.kv_slot_mapping, pr.kv_block_size, head=head,
                             ratio=ratio, overlap=overlap, state_width=sw, fmt=fmt)
        comp = np.zeros((pr.num_tokens, head), np.float32)
        kc = pr.k_cache.copy()
        assert oracle.forward_ex(sub, k_cache=kc, comp_out=comp, tokens=[t]) == 0
        want = (blk * sb + q % sb) * 2048 + ho + cols
        assert np.array_equal(comp[t], want.astype(np.float32)), (t, p)
        kvs = int(pr.kv_slot_mapping[t])
        tok, sc = _epilogue(fmt, comp[t], pr, p)
        got_tok, got_sc = _slot_bytes(kc, fmt, pr.kv_block_size, kvs)
        assert np.array_equal(got_tok, tok) and np.array_equal(got_sc, sc)
        other = np.ones(kc.shape, bool)
        blkv = other[kvs // pr.kv_block_size].reshape(-1)
        tb, sbt = SLOT[fmt]
        off = kvs % pr.kv_block_size
        blkv[off * tb:(off + 1) * tb] = False
        blkv[pr.kv_block_size * tb + off * sbt:pr.kv_block_size * tb + (off + 1) * sbt] = False
        assert np.array_equal(kc[other], pr.k_cache[other])   # nothing else written


def bt_blk(pr, r, q, sb):
    return int(pr.block_table[r, q // sb])


@pytest.mark.parametrize("head,ratio,overlap,fmt", [(128, 16, 1, 1), (512, 4, 1, 0), (128, 128, 0, 2),
                                                     (512, 128, 0, 0), (128, 2, 0, 1)])
def test_reblocking_invariance(head, ratio, overlap, fmt):
    """The same logical state rows paged with state blocks of 1, 2, 3, 4, 8, 16 and 64 rows (fresh
    block tables each time) give the same compressed vectors and the same k_cache bytes."""
    rng = np.random.default_rng([7, head, ratio, overlap, fmt])
    sw = head * (1 + overlap)
    n = (1 + overlap) * ratio
    lens = [int(rng.integers(n, 3 * n + 5)) for _ in range(3)] + [n - 1]
    logical = []
    for L in lens:
        rows = rng.standard_normal((L, 2 * sw)).astype(np.float32)
        rows[:, sw:] *= np.float32(2.0)
        logical.append(rows)
    ref = None
    for sb in (1, 2, 3, 4, 8, 16, 64):
        pr = _paged_problem(np.random.default_rng(sb), lens, head, ratio, overlap, fmt, sb, logical=logical)
        if ref is not None:   # same tokens, kv slots, rope table, weights and sentinel bytes
            pr.kv_slot_mapping, pr.k_cache, pr.cos_sin, pr.rms_w = ref[2], ref[3], ref[4], ref[5]
        kc = pr.k_cache.copy()
        comp = np.zeros((pr.num_tokens, head), np.float32)
        assert oracle.forward_ex(pr, k_cache=kc, comp_out=comp) == 0
        if ref is None:
            ref = (kc, comp, pr.kv_slot_mapping, pr.k_cache, pr.cos_sin, pr.rms_w)
            assert len(_active(pr)) >= 4 and not np.array_equal(kc, pr.k_cache)
        else:
            assert np.array_equal(comp, ref[1]), sb
            assert np.array_equal(kc, ref[0]), sb


def _brute_comp(pr, t):
    """float64 column softmax and weighted sum of token t's window, from the definition."""
    p, r = int(pr.positions[t]), int(pr.token_to_req[t])
    head, ratio, sw, sb = pr.head, pr.ratio, pr.state_width, pr.state.shape[1]
    kv, sc = [], []
    for i, q in _window_rows(p, ratio, pr.overlap):
        if q < 0:
            continue
        row = pr.state[pr.block_table[r, q // sb], q % sb].astype(np.float64)
        ho = head if i >= ratio else 0
        kv.append(row[ho:ho + head])
        sc.append(row[sw + ho:sw + ho + head])
    kv, sc = np.array(kv), np.array(sc)
    w = np.exp(sc - sc.max(axis=0))
    return (w * kv).sum(axis=0) / w.sum(axis=0)


@pytest.mark.parametrize("head,ratio,overlap,fmt,sb", [
    (128, 1, 0, 1, 1), (128, 1, 1, 2, 3), (128, 2, 0, 1, 3), (128, 2, 1, 2, 1), (128, 8, 0, 2, 3),
    (128, 8, 1, 1, 8), (128, 16, 1, 1, 5), (512, 16, 1, 0, 3), (512, 8, 0, 0, 1)])
def test_brute_force_small_ratios(head, ratio, overlap, fmt, sb):
    """Random kv ~ N(0,1) and score ~ N(0,2): every compressed value is the float64 definition
    rounded to fp32 (within half an fp32 ulp, plus float64 noise); every active token's record
    is the epilogue of it in its own slot; no other byte of the k_cache changes. Each request
    starts at position 0, so with overlap its first window has `ratio` masked rows."""
    rng = np.random.default_rng([11, head, ratio, overlap, fmt, sb])
    n = (1 + overlap) * ratio
    lens = [int(rng.integers(n, 4 * n + 9)) for _ in range(4)]
    pr = _paged_problem(rng, lens, head, ratio, overlap, fmt, sb, kv_bs=3)
    # a few padded tokens, tokens without a kv slot and negative positions: all inactive
    T = pr.num_tokens
    pr.slot_mapping[rng.choice(T, 3, replace=False)] = -1
    pr.kv_slot_mapping[rng.choice(T, 3, replace=False)] = -1
    kc = pr.k_cache.copy()
    comp = np.zeros((T, head), np.float32)
    assert oracle.forward_ex(pr, k_cache=kc, comp_out=comp) == 0
    act = _active(pr)
    assert len(act) >= 4
    written = np.zeros(kc.shape, bool)
    for t in act:
        ref = _brute_comp(pr, t)
        ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
        err = np.abs(comp[t].astype(np.float64) - ref)
        assert np.all(err <= 0.5 * ulp * (1 + 1e-6) + 1e-300), (t, float((err / ulp).max()))
        kvs = int(pr.kv_slot_mapping[t])
        tok, sc = _epilogue(fmt, comp[t], pr, int(pr.positions[t]))
        got_tok, got_sc = _slot_bytes(kc, fmt, pr.kv_block_size, kvs)
        assert np.array_equal(got_tok, tok) and np.array_equal(got_sc, sc), t
        tb, sbt = SLOT[fmt]
        bs, off = pr.kv_block_size, kvs % pr.kv_block_size
        wv = written[kvs // bs].reshape(-1)
        wv[off * tb:(off + 1) * tb] = True
        wv[bs * tb + off * sbt:bs * tb + (off + 1) * sbt] = True
    assert np.array_equal(kc[~written], pr.k_cache[~written])
    inactive = np.setdiff1d(np.arange(T), act)
    assert not comp[inactive].any()


def test_negative_positions_are_inactive_any_ratio():
    """p < 0 never stores, whatever the ratio ((p + 1) % ratio can be 0 for p = -1 in C)."""
    rng = np.random.default_rng(12)
    for ratio, overlap in ((1, 0), (4, 1), (16, 1), (128, 0)):
        pr = _paged_problem(rng, [2 * ratio * (1 + overlap)], 128, ratio, overlap, 1, 4)
        pr.positions = pr.positions - (2 * ratio * (1 + overlap) + 3)    # every position negative
        kc = pr.k_cache.copy()
        assert oracle.forward_ex(pr, k_cache=kc) == 0
        assert np.array_equal(kc, pr.k_cache)
