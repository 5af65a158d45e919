"""Seeded random configurations of SnapKV++ compression (GQA ratio, window, ragged lengths
including ones the keep covers whole, pooling kernel incl. the per-sequence one, keep) checked
against the oracle: scores, kept positions and the gathered rows of every (unit, KV head)."""
import numpy as np
import pytest

from tests import test_gpu_snapkv as T

pytestmark = pytest.mark.gpu


def _config(seed):
    r = np.random.default_rng(3000 + seed)
    gqa = int(r.choice([1, 2, 4, 8]))
    window = int(r.integers(1, 256 // gqa + 1))
    n_seq, n_kv = int(r.integers(1, 4)), int(r.integers(1, 3))
    max_len = int(r.integers(window + 2, 10000))
    lens = [int(x) for x in r.integers(window + 1, max_len + 1, size=n_seq)]
    lens[0] = max_len
    kernel = int(r.choice([0, 1, 3, 5, 7, 9, 15, 21, 31]))
    keep = int(r.integers(window + 1, max(window + 2, max_len)))
    return n_seq, n_kv, gqa, window, lens, kernel, keep


@pytest.mark.parametrize("seed", range(24))
def test_snapkv_random_configuration(seed):
    rkv = T._lib()
    n_seq, n_kv, gqa, window, lens, kernel, keep = _config(seed)
    wl, x = T._inputs(n_seq, n_kv, gqa, lens, window, seed=4000 + seed, needles=4)
    k_out, v_out, kept, out_len, scores = T._run(rkv, x, window, kernel, keep)
    for u in range(n_seq):
        for g in range(n_kv):
            T._check_unit(x, u, g, gqa, window, kernel, keep, k_out, v_out, kept, out_len,
                          scores, tag=f"seed {seed} unit {u} kv {g}")
