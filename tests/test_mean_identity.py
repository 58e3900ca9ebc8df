"""The identity the kernels' mean relies on (CPU): for N a power of two, the float32
product x * (1/N) equals the float32 quotient x / N bit for bit -- 1/N is exact, so both
are the one real number x/N rounded once -- over random bit patterns, subnormals, zeros,
infinities and the largest values; NaNs stay NaNs.  For other N the two can differ,
which is why the kernels divide there."""
import numpy as np
import pytest


def patterns(n, seed):
    rng = np.random.default_rng(seed)
    u = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x007FFFFF, 0x00800000, 0x7F7FFFFF,
                        0xFF7FFFFF, 0x7F800000, 0xFF800000, 0x7FC00000, 0x3F800000, 0x00000003], np.uint32)
    return np.concatenate([u, special]).view(np.float32)


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 32, 64])
def test_power_of_two_mean_multiply_equals_division(N):
    x = patterns(1_000_000, N)
    with np.errstate(all="ignore"):
        q = x / np.float32(N)
        p = x * (np.float32(1) / np.float32(N))
    nan = np.isnan(q)
    assert np.array_equal(nan, np.isnan(p))
    assert np.array_equal(q[~nan].view(np.uint32), p[~nan].view(np.uint32))


def test_other_n_can_differ():
    x = patterns(1_000_000, 6)
    with np.errstate(all="ignore"):
        q = x / np.float32(6)
        p = x * (np.float32(1) / np.float32(6))
    ok = ~np.isnan(q)
    assert (q[ok].view(np.uint32) != p[ok].view(np.uint32)).any()
