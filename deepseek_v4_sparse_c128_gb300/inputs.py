"""Seeded synthetic inputs for the C128 compress -> RMSNorm -> FP8/RoPE -> paged-store op.

This module only draws and lays out data; it holds none of the op's arithmetic. Both the
CUDA path and the CPU oracle consume what it returns, so it is the one piece of code they
share.

Shapes and value distributions follow the DeepSeek-V4 C128 layout described in
"optimize the compressor 128 split cutedsl kernel" (vLLM PR #44230, Summary and
Validation) and the cache-layout docstrings of
``vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache``
(``_fused_kv_compress_norm_rope_insert_sparse_attn``):

* state cache ``[num_blocks, 8, 1024]`` fp32, a row is ``kv[0:512] | score[512:1024]``;
  kv ~ N(0, 1), score ~ N(0, sigma=2);
* ``block_table [num_reqs, max_blocks]`` int32 (every entry a valid block id);
* ``positions``, ``slot_mapping``, ``kv_slot_mapping`` int64, ``token_to_req_indices`` int32;
* ``rms_w = 1 + 0.1 N(0, 1)`` fp32 [512], ``eps = 1e-6``;
* ``cos_sin_cache [max_pos, 64]`` fp32, cos in [0, 32), sin in [32, 64), rope theta 10000;
* ``k_cache [num_kv_blocks, kv_block_size, 584]`` uint8, pre-filled with random sentinel bytes.

Five workloads (the tiny, decode, mixed, varlen and all-boundary sweep cases) are built by
``make_problem``. Large state caches can be drawn on a CUDA device with torch's Philox
generator (``state_device="cuda"``); everything else is drawn with numpy's PCG64.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

HEAD = 512            # head size (nope 448 + rope 64)
STATE_WIDTH = 512     # kv columns; the score columns follow them
ROW = 2 * STATE_WIDTH  # fp32 values per state-cache row
STATE_BLOCK = 8       # rows per state-cache block
RATIO = 128           # compress ratio: rows per window
ROPE = 64
TOKEN_BYTES = 584     # 448 fp8 + 64 bf16 (= 576 B) + 8 scale bytes per token

SWEEP_TOKENS = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192, 16374)
# slot bytes (token data + scales) of each cache format
SLOT_BYTES = {0: 576 + 8, 1: 128 + 4, 2: 64 + 4}
CONFIG_SEEDS = {"tiny": 0, "decode": 1, "mixed": 2, "varlen": 3, "sweep": 4, "varlen16k": 5}


@dataclasses.dataclass
class Problem:
    """One call's worth of inputs. ``state`` is a numpy array or a torch tensor."""

    name: str
    token_to_req: np.ndarray      # int32 [T]
    positions: np.ndarray         # int64 [T]
    slot_mapping: np.ndarray      # int64 [T]
    block_table: np.ndarray       # int32 [R, MB]
    state: object                 # float32 [NB, 8, 1024] (numpy or torch)
    rms_w: np.ndarray             # float32 [512]
    eps: float
    cos_sin: np.ndarray           # float32 [MP, 64]
    k_cache: np.ndarray           # uint8 [NKB, bs, slot bytes]
    kv_slot_mapping: np.ndarray   # int64 [T]
    kv_block_size: int
    # configuration (defaults: the C128 sparse-attention compressor)
    head: int = 512               # 512 (sparse attention) or 128 (indexer)
    ratio: int = 128              # compress ratio
    overlap: int = 0              # 1: windows of 2*ratio rows, the newer half at +head
    state_width: int = 512        # kv columns of a state row; as many score columns follow
    fmt: int = 0                  # cache format: 0 sparse FP8 + bf16 rope, 1 indexer FP8, 2 indexer MXFP4

    @property
    def num_tokens(self) -> int:
        return int(self.positions.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.state.shape[0]) if self.state is not None else 0


def _cos_sin_cache(max_pos: int, theta: float = 10000.0) -> np.ndarray:
    """GPT-J style rope table: angle(pos, j) = pos * theta^(-2j/64), computed in fp64."""
    j = np.arange(ROPE // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / ROPE)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _draw_state_numpy(rng: np.random.Generator, num_blocks: int) -> np.ndarray:
    st = np.empty((num_blocks, STATE_BLOCK, ROW), dtype=np.float32)
    st[..., :STATE_WIDTH] = rng.standard_normal((num_blocks, STATE_BLOCK, STATE_WIDTH), dtype=np.float32)
    st[..., STATE_WIDTH:] = rng.standard_normal((num_blocks, STATE_BLOCK, STATE_WIDTH), dtype=np.float32)
    st[..., STATE_WIDTH:] *= np.float32(2.0)
    return st


def draw_state(seed: int, num_blocks: int, device: str = "cpu"):
    """State cache ``[num_blocks, 8, 1024]``: kv ~ N(0,1) then score ~ N(0,2) in every row.
    ``device="none"`` skips the draw (metadata-only problems)."""
    if device == "none":
        return None
    if device == "cpu":
        return _draw_state_numpy(np.random.default_rng([seed, 0x5EED]), num_blocks)
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 17)
    st = torch.empty((num_blocks, STATE_BLOCK, ROW), dtype=torch.float32, device=device)
    # draw in slabs so the temporary stays small for multi-GB caches
    slab = 4096
    for b0 in range(0, num_blocks, slab):
        b1 = min(num_blocks, b0 + slab)
        v = torch.randn((b1 - b0, STATE_BLOCK, ROW), generator=g, device=device, dtype=torch.float32)
        v[..., STATE_WIDTH:] *= 2.0
        st[b0:b1] = v
    return st


def _rms_w(rng: np.random.Generator) -> np.ndarray:
    return (1.0 + 0.1 * rng.standard_normal(HEAD)).astype(np.float32)


def _k_cache(rng: np.random.Generator, num_kv_blocks: int, bs: int) -> np.ndarray:
    return rng.integers(0, 256, size=(num_kv_blocks, bs, TOKEN_BYTES), dtype=np.uint8)


def _state_slot(block_table: np.ndarray, req: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """The state-cache slot a token's own row lives in (only its sign matters to the op)."""
    blk = block_table[req, pos // STATE_BLOCK].astype(np.int64)
    return blk * STATE_BLOCK + pos % STATE_BLOCK


def _tiny(seed: int, state_device: str) -> Problem:
    rng = np.random.default_rng(seed)
    R, MB, NB = 4, 64, 64
    bt = np.stack([rng.permutation(NB) for _ in range(R)]).astype(np.int32)
    req = np.arange(R, dtype=np.int32)
    pos = np.array([127, 255, 383, 511], dtype=np.int64)
    kv_slot = rng.permutation(8)[:4].astype(np.int64)
    return Problem("tiny", req, pos, _state_slot(bt, req, pos), bt, draw_state(seed, NB, state_device),
                   _rms_w(rng), 1e-6, _cos_sin_cache(512), _k_cache(rng, 4, 2), kv_slot, 2)


def _windows_at_boundary(rng, n_tok, nb_pool, mb):
    """Each token its own request at p = 128k-1; its 16 window blocks are a distinct chunk of a
    shuffled pool; the other block-table entries hold random (valid) ids."""
    k = rng.integers(1, 65, size=n_tok)
    pos = (RATIO * k - 1).astype(np.int64)
    bt = rng.integers(0, nb_pool, size=(n_tok, mb), dtype=np.int64).astype(np.int32)
    pool = rng.permutation(nb_pool)
    first = (pos - (RATIO - 1)) // STATE_BLOCK
    for t in range(n_tok):
        bt[t, first[t]:first[t] + RATIO // STATE_BLOCK] = pool[16 * t:16 * t + 16]
    return pos, bt


def _decode(seed: int, state_device: str) -> Problem:
    rng = np.random.default_rng(seed)
    T, MB, NB = 128, 1024, 2048
    pos, bt = _windows_at_boundary(rng, T, NB, MB)
    req = np.arange(T, dtype=np.int32)
    NKB, bs = 96, 2
    kv_slot = rng.permutation(NKB * bs)[:T].astype(np.int64)
    return Problem("decode", req, pos, _state_slot(bt, req, pos), bt, draw_state(seed, NB, state_device),
                   _rms_w(rng), 1e-6, _cos_sin_cache(8192), _k_cache(rng, NKB, bs), kv_slot, bs)


def _mixed(seed: int, state_device: str) -> Problem:
    rng = np.random.default_rng(seed)
    R, per, MB, NB = 256, 16, 1024, 4096
    T = R * per
    req = np.repeat(np.arange(R, dtype=np.int32), per)
    pos = rng.integers(0, 8192, size=T).astype(np.int64)
    bt = rng.integers(0, NB, size=(R, MB)).astype(np.int32)
    slot = _state_slot(bt, req, pos)
    pad = rng.choice(T, size=int(round(0.1 * T)), replace=False)
    slot[pad] = -1
    bs = 2
    NKB = T // bs
    kv_slot = rng.permutation(T).astype(np.int64)
    return Problem("mixed", req, pos, slot, bt, draw_state(seed, NB, state_device),
                   _rms_w(rng), 1e-6, _cos_sin_cache(8192), _k_cache(rng, NKB, bs), kv_slot, bs)


def _varlen_from_lengths(name, seed, lens, state_device, rng) -> Problem:
    lens = np.asarray(lens, dtype=np.int64)
    R = lens.shape[0]
    nblk = (lens + STATE_BLOCK - 1) // STATE_BLOCK
    NB = int(nblk.sum())
    MB = int(nblk.max())
    pool = rng.permutation(NB)
    bt = rng.integers(0, NB, size=(R, MB)).astype(np.int32)
    off = 0
    for r in range(R):
        bt[r, :nblk[r]] = pool[off:off + nblk[r]]
        off += nblk[r]
    req = np.repeat(np.arange(R, dtype=np.int32), lens)
    pos = np.concatenate([np.arange(n, dtype=np.int64) for n in lens])
    slot = _state_slot(bt, req, pos)
    bs = 64
    nwin = lens // RATIO
    kvblk_per_req = (nwin + bs - 1) // bs
    NKB = int(kvblk_per_req.sum())
    kvpool = rng.permutation(NKB)
    kv_slot = np.full(pos.shape[0], -1, dtype=np.int64)
    tok0 = np.concatenate([[0], np.cumsum(lens)[:-1]])
    koff = 0
    for r in range(R):
        kb = kvpool[koff:koff + kvblk_per_req[r]]
        koff += kvblk_per_req[r]
        k = np.arange(nwin[r])
        kv_slot[tok0[r] + RATIO * (k + 1) - 1] = kb[k // bs].astype(np.int64) * bs + k % bs
    max_pos = int(lens.max())
    return Problem(name, req, pos, slot, bt, draw_state(seed, NB, state_device),
                   _rms_w(rng), 1e-6, _cos_sin_cache(max_pos), _k_cache(rng, max(NKB, 1), bs), kv_slot, bs)


def _varlen(seed: int, state_device: str) -> Problem:
    rng = np.random.default_rng(seed)
    lens = rng.integers(128, 16385, size=32)
    return _varlen_from_lengths("varlen", seed, lens, state_device, rng)


def _varlen16k(seed: int, state_device: str) -> Problem:
    """Same recipe with the drawn lengths rescaled so they total about 16k tokens."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(128, 16385, size=32).astype(np.float64)
    lens = np.maximum(128, np.floor(lens * (16384.0 / lens.sum()))).astype(np.int64)
    return _varlen_from_lengths("varlen16k", seed, lens, state_device, rng)


def _sweep(seed: int, T: int, state_device: str) -> Problem:
    rng = np.random.default_rng([seed, T])
    MB = 1024
    NB = 16 * T
    pos, bt = _windows_at_boundary(rng, T, NB, MB)
    req = np.arange(T, dtype=np.int32)
    bs = 2
    NKB = (T + bs - 1) // bs
    kv_slot = rng.permutation(NKB * bs)[:T].astype(np.int64)
    return Problem(f"sweep{T}", req, pos, _state_slot(bt, req, pos), bt, draw_state(seed * 100003 + T, NB, state_device),
                   _rms_w(rng), 1e-6, _cos_sin_cache(8192), _k_cache(rng, NKB, bs), kv_slot, bs)


def make_problem(name: str, seed: Optional[int] = None, tokens: Optional[int] = None,
                 state_device: str = "cpu") -> Problem:
    """Build one of the named workloads. ``tokens`` selects the sweep point."""
    if seed is None:
        seed = CONFIG_SEEDS["sweep" if name.startswith("sweep") else name]
    if name == "tiny":
        return _tiny(seed, state_device)
    if name == "decode":
        return _decode(seed, state_device)
    if name == "mixed":
        return _mixed(seed, state_device)
    if name == "varlen":
        return _varlen(seed, state_device)
    if name == "varlen16k":
        return _varlen16k(seed, state_device)
    if name.startswith("sweep"):
        T = tokens if tokens is not None else int(name[5:] or 16374)
        return _sweep(seed, T, state_device)
    raise ValueError(f"unknown workload {name!r}")


def draw_state_rows(seed: int, num_blocks: int, block: int, state_width: int, device: str = "cpu"):
    """State cache [num_blocks, block, 2*state_width]: kv ~ N(0,1) then score ~ N(0,2) in every row."""
    if device == "none":
        return None
    if device == "cpu":
        rng = np.random.default_rng([seed, 0x5EED, state_width])
        st = rng.standard_normal((num_blocks, block, 2 * state_width), dtype=np.float32)
        st[..., state_width:] *= np.float32(2.0)
        return st
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 29)
    st = torch.randn((num_blocks, block, 2 * state_width), generator=g, device=device, dtype=torch.float32)
    st[..., state_width:] *= 2.0
    return st


def prefill_problem(name: str, seed: int, num_reqs: int, min_len: int, max_len: int, head: int, ratio: int,
                    overlap: int, fmt: int, state_block: int = 8, kv_block_size: int = 64,
                    state_device: str = "cpu", decode_tail: int = 0) -> Problem:
    """Requests with every position 0..len-1 present (window ends active: every `ratio`-th token),
    request-major, blocks from a shuffled pool; optionally `decode_tail` extra one-token requests
    at window ends. State width is head * (1 + overlap)."""
    rng = np.random.default_rng([seed, ratio, head, fmt])
    sw = head * (1 + overlap)
    lens = rng.integers(min_len, max_len + 1, size=num_reqs).astype(np.int64)
    if decode_tail:
        k = rng.integers(1, 65, size=decode_tail) if ratio >= 128 else rng.integers(8, 512, size=decode_tail)
        lens = np.concatenate([lens, ratio * k])
    R = lens.shape[0]
    nblk = (lens + state_block - 1) // state_block
    NB, MB = int(nblk.sum()), int(nblk.max())
    pool = rng.permutation(NB)
    bt = rng.integers(0, NB, size=(R, MB)).astype(np.int32)
    off = 0
    for r in range(R):
        bt[r, :nblk[r]] = pool[off:off + nblk[r]]
        off += nblk[r]
    if decode_tail:   # the one-token requests carry only their last position
        req = np.concatenate([np.repeat(np.arange(num_reqs, dtype=np.int32), lens[:num_reqs]),
                              np.arange(num_reqs, R, dtype=np.int32)])
        pos = np.concatenate([np.concatenate([np.arange(n, dtype=np.int64) for n in lens[:num_reqs]]),
                              lens[num_reqs:] - 1])
    else:
        req = np.repeat(np.arange(R, dtype=np.int32), lens)
        pos = np.concatenate([np.arange(n, dtype=np.int64) for n in lens])
    slot = _state_slot_blocks(bt, req, pos, state_block)
    active = (pos + 1) % ratio == 0
    A = int(active.sum())
    NKB = max(1, -(-A // kv_block_size))
    kv_slot = np.full(pos.shape[0], -1, dtype=np.int64)
    kv_slot[np.nonzero(active)[0]] = rng.permutation(NKB * kv_block_size)[:A]
    max_pos = int(pos.max()) + 1
    return Problem(name, req, pos, slot, bt, draw_state_rows(seed, NB, state_block, sw, state_device),
                   _rms_w(rng)[:head].copy(), 1e-6, _cos_sin_cache(max_pos),
                   rng.integers(0, 256, size=(NKB, kv_block_size, SLOT_BYTES[fmt]), dtype=np.uint8), kv_slot,
                   kv_block_size, head=head, ratio=ratio, overlap=overlap, state_width=sw, fmt=fmt)


def _state_slot_blocks(block_table, req, pos, state_block):
    blk = block_table[req, pos // state_block].astype(np.int64)
    return blk * state_block + pos % state_block


def make_next_problem(name: str, state_device: str = "cpu", scale: int = 1) -> Problem:
    """Workloads for the other configurations: C4 sparse attention (head 512, ratio 4, overlap),
    the indexer (head 128) with FP8 or MXFP4 caches at ratio 4 with overlap and at ratio 128."""
    spec = {
        "c4_sparse": (512, 4, 1, 0), "idx_c4_fp8": (128, 4, 1, 1), "idx_c4_mxfp4": (128, 4, 1, 2),
        "idx_c128_fp8": (128, 128, 0, 1), "idx_c128_mxfp4": (128, 128, 0, 2),
    }[name]
    head, ratio, overlap, fmt = spec
    if ratio == 4:
        return prefill_problem(name, 6, 8 * scale, 5, 1024, head, ratio, overlap, fmt, state_device=state_device,
                               decode_tail=16 * scale)
    return prefill_problem(name, 7, 4 * scale, 128, 8192, head, ratio, overlap, fmt, state_device=state_device,
                           decode_tail=64 * scale)


def random_problem(seed: int, num_tokens: int, num_reqs: int, max_blocks: int, num_blocks: int,
                   kv_block_size: int, active_frac: float = 0.5, pad_frac: float = 0.1,
                   kv_drop_frac: float = 0.05, max_pos: Optional[int] = None) -> Problem:
    """A small randomised case: random requests, positions (about ``active_frac`` of them at a
    window end), padded tokens (slot -1), tokens without a kv slot (kv slot -1), negative
    positions, iid block-table entries (blocks may alias across windows)."""
    rng = np.random.default_rng(seed)
    T = num_tokens
    max_p = max_blocks * STATE_BLOCK - 1
    req = rng.integers(0, num_reqs, size=T).astype(np.int32)
    k = rng.integers(1, max_p // RATIO + 1, size=T)
    pos = np.where(rng.random(T) < active_frac, RATIO * k - 1, rng.integers(0, max_p + 1, size=T)).astype(np.int64)
    neg = rng.random(T) < 0.02
    pos[neg] = -1 - rng.integers(0, 300, size=int(neg.sum()))
    bt = rng.integers(0, num_blocks, size=(num_reqs, max_blocks)).astype(np.int32)
    slot = np.where(pos >= 0, 1 + rng.integers(0, 1 << 20, size=T), 0).astype(np.int64)
    slot[rng.random(T) < pad_frac] = -1
    NKB = max(1, -(-T // kv_block_size))
    kv_slot = rng.permutation(NKB * kv_block_size)[:T].astype(np.int64)
    kv_slot[rng.random(T) < kv_drop_frac] = -1
    mp = max_pos if max_pos is not None else max_blocks * STATE_BLOCK
    return Problem(f"random{seed}", req, pos, slot, bt, draw_state(seed, num_blocks, "cpu"),
                   _rms_w(rng), 1e-6, _cos_sin_cache(mp), _k_cache(rng, NKB, kv_block_size), kv_slot,
                   kv_block_size)
