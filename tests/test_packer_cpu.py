"""The host-side packer (varlen_pack_sequences) against the oracle's packing
loops: the same packs, index for index, and the same padding rate (CPU only:
the packer does no GPU work, so the library loads and runs here)."""
import numpy as np
import pytest

import oracle
from selective_ssm_packed_gb300 import binding


@pytest.fixture(scope="module")
def lib():
    from selective_ssm_packed_gb300 import build
    build.build()
    return binding.lib()


def _lengths(seed, n, size, median=800):
    rng = np.random.default_rng(seed)
    L = np.clip(np.exp(rng.normal(np.log(median), 1.0, n)), 1, size).astype(np.int32)
    L[rng.choice(n, max(1, n // 100), replace=False)] = 0  # a few empty sequences
    return L


@pytest.mark.parametrize("seed,n,size,window", [(1, 1, 4096, 1), (2, 500, 4096, 64), (3, 3000, 4096, 1000),
                                                (4, 2000, 8192, 7), (5, 777, 2048, 777)])
def test_packer_matches_the_oracle(lib, seed, n, size, window):
    L = _lengths(seed, n, size)
    for method, ref in (("sequential", oracle.pack_sequential(L.tolist(), size)),
                        ("local_greedy", oracle.pack_local_greedy(L.tolist(), size, window))):
        packs, pad = binding.pack_sequences(L, size, method, window)
        assert [p.tolist() for p in packs] == ref, method
        assert pad == pytest.approx(oracle.padding_rate(L.tolist(), ref, size), abs=1e-15)


def test_local_greedy_pads_less_than_sequential_on_the_workload_mix(lib):
    # the article's observation (19.1 % -> 0.46 % on its data) on the bench's length mix
    L = _lengths(6, 20000, 4096)
    _, seq = binding.pack_sequences(L, 4096, "sequential")
    _, gr = binding.pack_sequences(L, 4096, "local_greedy", 1000)
    assert gr < seq and gr < 0.02


def test_packer_rejects_bad_arguments(lib):
    with pytest.raises(binding.VssmError):
        binding.pack_sequences([5, 9000], 4096, "sequential")       # longer than a pack
    with pytest.raises(binding.VssmError):
        binding.pack_sequences([5, -1], 4096, "local_greedy", 10)   # negative length
    with pytest.raises(binding.VssmError):
        binding.pack_sequences([5, 1], 4096, "local_greedy", 0)     # window
    assert binding.pack_sequences([], 4096, "sequential") == ([], 0.0)
