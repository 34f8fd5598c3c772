"""Host-side logic of bench.py that needs no GPU."""
import math
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_profile_stride_is_coprime_with_the_pool():
    # sampled steps must visit every entry of the input pool
    for pool in range(1, 130):
        k = bench.profile_stride(pool)
        assert k >= bench.PROFILE_EVERY
        assert math.gcd(k, pool) == 1
        assert sorted({(s * k) % pool for s in range(pool)}) == list(range(pool))
