"""Pins the oracle's Philox4x32-10 bit stream to an independent implementation
of the same generator: cuRAND's host-side PHILOX4_32_10 generator (it runs on
the CPU, no GPU needed). Its output block i, for a 64-bit seed s, is the
generator applied to counter (0, 0, i, 0) with key (s mod 2^32, s div 2^32);
every word of 2^14 blocks must equal the oracle's for the same counter and key.
A wrong round multiplier, a swapped output word, a missed key bump or a wrong
Weyl constant changes essentially every word, so it fails here (the
statistical pins in test_oracle_sampling would not see it)."""
import ctypes
import glob
import os

import numpy as np
import pytest

from oracle.sampling import philox4x32_10

CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161  # curand.h


def _curand():
    cands = ["/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"]
    try:
        import nvidia  # pip-packaged CUDA libraries next to torch, if any
        for p in nvidia.__path__:
            cands += sorted(glob.glob(os.path.join(p, "curand", "lib", "libcurand.so*")))
    except ImportError:
        pass
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    pytest.skip("libcurand not found")


def curand_host_words(seed, n):
    lib = _curand()
    gen = ctypes.c_void_p()
    st = lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10)
    if st != 0:
        pytest.skip(f"curandCreateGeneratorHost failed ({st})")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out.astype(np.uint64)


@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_philox_matches_curand_host_generator(seed):
    n_blocks = 1 << 14
    got = curand_host_words(seed, 4 * n_blocks).reshape(-1, 4)
    ctr = np.zeros((n_blocks, 4), dtype=np.uint64)
    ctr[:, 2] = np.arange(n_blocks, dtype=np.uint64)
    want = philox4x32_10(ctr, (seed & 0xFFFFFFFF, seed >> 32))
    assert np.array_equal(want, got)


def test_a_planted_output_word_swap_is_caught():
    seed = 12345
    got = curand_host_words(seed, 64).reshape(-1, 4)
    ctr = np.zeros((16, 4), dtype=np.uint64)
    ctr[:, 2] = np.arange(16, dtype=np.uint64)
    want = philox4x32_10(ctr, (seed, 0))
    assert np.array_equal(want, got)
    assert not np.array_equal(want[:, [1, 0, 2, 3]], got)
