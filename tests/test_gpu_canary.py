"""Out-of-bounds writes: k_cache and the fp32 export each sit inside a larger device buffer filled
with random canary bytes, for every kernel path (cluster-split, one CTA per token, planning pass +
window queue, the small-window ring, the ratio-128 indexer ring, the gather kernel). After the
call, every canary byte must be unchanged and the bytes inside must match the oracle."""
import numpy as np
import pytest

from deepseek_v4_sparse_c128_gb300 import inputs
from gpu_util import NAN_BITS, check_against_oracle, check_against_oracle_ex, to_device

pytestmark = pytest.mark.gpu

GUARD = 4096  # canary bytes before and after (a multiple of 16, so alignment is kept)


@pytest.fixture(scope="module")
def binding():
    from deepseek_v4_sparse_c128_gb300 import binding as b
    from deepseek_v4_sparse_c128_gb300 import build
    build.build()
    b.load()
    return b


def _guarded(arr: np.ndarray, seed: int):
    """A device buffer of canary bytes with `arr` copied into its middle; returns (buffer, view)."""
    import torch
    nbytes = arr.nbytes
    rng = np.random.default_rng(seed)
    host = rng.integers(0, 256, size=nbytes + 2 * GUARD, dtype=np.uint8)
    host[GUARD:GUARD + nbytes] = arr.view(np.uint8).reshape(-1)
    buf = torch.from_numpy(host).cuda()
    view = buf[GUARD:GUARD + nbytes].view(torch.from_numpy(arr[:0]).dtype).view(arr.shape)
    return buf, view, host


def _canaries_intact(buf, host, nbytes):
    got = buf.cpu().numpy()
    assert np.array_equal(got[:GUARD], host[:GUARD]), "bytes before the buffer changed"
    assert np.array_equal(got[GUARD + nbytes:], host[GUARD + nbytes:]), "bytes after the buffer changed"


@pytest.mark.parametrize("name,tokens", [("decode", None), ("tiny", None), ("mixed", None), ("sweep", 300),
                                         ("sweep", 2000)])
def test_c128_paths_write_inside_their_buffers(binding, name, tokens):
    import torch
    p = inputs.make_problem(name, tokens=tokens) if tokens else inputs.make_problem(name)
    d = to_device(p)
    kbuf, d["k_cache"], khost = _guarded(p.k_cache, 1)
    comp0 = np.full((p.num_tokens, 512), NAN_BITS, np.uint32).view(np.float32)
    cbuf, comp_out, chost = _guarded(comp0, 2)
    binding.compress_norm_rope_store(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                     d["state"], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"], d["kv_slot_mapping"],
                                     p.kv_block_size, comp_out=comp_out)
    torch.cuda.synchronize()
    assert binding.device_errors(clear=True) == 0
    _canaries_intact(kbuf, khost, p.k_cache.nbytes)
    _canaries_intact(cbuf, chost, comp0.nbytes)
    check_against_oracle(p, d["k_cache"].cpu().numpy(), comp_out.cpu().numpy(), threads=16)


@pytest.mark.parametrize("name", ["c4_sparse", "idx_c4_mxfp4", "idx_c128_fp8"])
def test_other_configurations_write_inside_their_buffers(binding, name):
    import torch
    p = inputs.make_next_problem(name)
    d = to_device(p)
    kbuf, d["k_cache"], khost = _guarded(p.k_cache, 3)
    comp0 = np.full((p.num_tokens, p.head), NAN_BITS, np.uint32).view(np.float32)
    cbuf, comp_out, chost = _guarded(comp0, 4)
    cfg = binding.config(p.head, p.ratio, p.overlap, p.state_width, p.fmt)
    binding.compress_norm_rope_store_ex(cfg, d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                        d["state"], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
                                        d["kv_slot_mapping"], p.kv_block_size, comp_out=comp_out)
    torch.cuda.synchronize()
    assert binding.device_errors(clear=True) == 0
    _canaries_intact(kbuf, khost, p.k_cache.nbytes)
    _canaries_intact(cbuf, chost, comp0.nbytes)
    check_against_oracle_ex(p, d["k_cache"].cpu().numpy(), comp_out.cpu().numpy(), threads=16)


def test_gather_kernel_writes_inside_its_buffers(binding):
    """Head 128 with a state block that is not a multiple of 8 rows: the gather kernel."""
    import torch
    p = inputs.prefill_problem("canary_gather", 41, 4, 5, 2000, 128, 128, 0, 2, state_block=4, kv_block_size=16,
                               decode_tail=6)
    d = to_device(p)
    kbuf, d["k_cache"], khost = _guarded(p.k_cache, 5)
    cfg = binding.config(p.head, p.ratio, p.overlap, p.state_width, p.fmt)
    comp0 = np.full((p.num_tokens, p.head), NAN_BITS, np.uint32).view(np.float32)
    cbuf, comp_out, chost = _guarded(comp0, 6)
    binding.compress_norm_rope_store_ex(cfg, d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                        d["state"], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
                                        d["kv_slot_mapping"], p.kv_block_size, comp_out=comp_out)
    torch.cuda.synchronize()
    assert binding.device_errors(clear=True) == 0
    _canaries_intact(kbuf, khost, p.k_cache.nbytes)
    _canaries_intact(cbuf, chost, comp0.nbytes)
    check_against_oracle_ex(p, d["k_cache"].cpu().numpy(), comp_out.cpu().numpy(), threads=16)
