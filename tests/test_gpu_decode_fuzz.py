"""Seeded random configurations of the hybrid decode (shapes, GQA ratio, budget, page, kept
channels, ragged lengths incl. dense ones), each checked against the oracle in both shared-memory
layouts."""
import numpy as np
import pytest

from tests import test_gpu_decode as T

pytestmark = pytest.mark.gpu


def _config(seed):
    r = np.random.default_rng(1000 + seed)
    gqa = int(r.choice([1, 2, 4, 8]))
    page = int(r.choice([1, 2, 4, 8, 16, 32, 64]))
    budget = 2 * page * int(r.integers(1, max(2, 1024 // page)))   # even, >= one page per half
    channels = int(r.integers(1, 129))
    n, n_kv = int(r.integers(1, 4)), int(r.integers(1, 3))
    cap = int(r.integers(64, 6000))
    lens = [int(x) for x in r.integers(1, cap + 1, size=n)]
    if seed % 3 == 0:
        lens[0] = min(cap, budget)          # exactly at the dense boundary
    return n, n_kv, gqa, lens, cap, budget, page, channels


@pytest.mark.parametrize("seed", range(40))
@pytest.mark.parametrize("layout", [1, 2], ids=["ordinary", "wide"])
def test_decode_random_configuration(seed, layout):
    rkv = T._lib()
    n, n_kv, gqa, lens, cap, budget, page, channels = _config(seed)
    rkv.rkv_testing_decode_layout(layout)
    try:
        T._hybrid_case(n, n_kv, gqa, lens, cap, budget, page, channels, seed=2000 + seed,
                       steps=1)
    finally:
        rkv.rkv_testing_decode_layout(0)
