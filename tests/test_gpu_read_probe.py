"""The read-bandwidth probe reads every byte it is given: the XOR word it returns equals the XOR
of the buffer's 32-bit words (numpy), for every load depth and launch shape, on buffers with a
ragged tail and on buffers smaller than one wave of loads."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _xor_words(a: np.ndarray) -> int:
    return int(np.bitwise_xor.reduce(a.view(np.uint32).reshape(-1))) if a.size else 0


@pytest.mark.parametrize("nbytes", [16, 48, 4096 + 16, 64 * 1024 * 1024 + 16 * 7])
@pytest.mark.parametrize("threads,ctas,loads", [(32, 1, 1), (256, 2, 2), (512, 2, 4), (1024, 1, 8), (512, 4, 8)])
def test_read_probe_xor_matches_numpy(nbytes, threads, ctas, loads):
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    rng = np.random.default_rng(nbytes + 7 * threads + loads)
    host = rng.integers(0, 2**32, size=nbytes // 4, dtype=np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.read_probe(buf, word, threads_per_cta=threads, ctas_per_sm=ctas, loads_in_flight=loads)
    torch.cuda.synchronize()
    assert int(word.cpu().numpy().view(np.uint32)[0]) == _xor_words(host)


def test_read_probe_twice_cancels():
    """Two passes over the same buffer XOR to zero: nothing outside the buffer is read into the word."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    buf = torch.randint(-2**31, 2**31 - 1, (3 * 1024 * 1024 + 4,), dtype=torch.int32, device="cuda")
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.read_probe(buf, word)
    binding.read_probe(buf, word)
    torch.cuda.synchronize()
    assert int(word.item()) == 0
