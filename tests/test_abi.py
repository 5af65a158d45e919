"""Host-side checks of the C ABI: the library builds, loads and exports every symbol that
include/*.h declares; the planner matches the oracle; invalid arguments are rejected on the host
before any launch. No GPU needed."""
import ctypes
import os
import re

import pytest

from oracle import rocketkv as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_kv_cache_snapkv_gb300 import _build, rkv
    _build.build()
    return rkv.load()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for hdr in sorted(os.listdir(inc)):
        if hdr.endswith(".h"):
            src = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, hdr)).read(), flags=re.S)
            names |= set(re.findall(r"\b(rkv_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name
    from sparse_kv_cache_snapkv_gb300 import rkv
    assert set(rkv.SYMBOLS) <= set(names)


@pytest.mark.parametrize("ctx", [300, 4096, 8192, 32768, 50000, 131072])
@pytest.mark.parametrize("budget", [256, 512, 1024, 4096])
def test_plan_matches_oracle(lib, ctx, budget):
    from sparse_kv_cache_snapkv_gb300 import rkv
    assert rkv.rkv_plan(ctx, budget) == O.plan(ctx, budget, 128)
    assert rkv.rkv_plan(ctx, budget, 128, 16, 128) == O.plan(ctx, budget, 128, 16, 128)


def test_plan_rejects(lib):
    out = [ctypes.c_int() for _ in range(4)]
    refs = [ctypes.byref(o) for o in out]
    assert lib.rkv_plan(4096, 255, 128, 0, 0, *refs) == 1      # odd budget
    assert lib.rkv_plan(4096, 256, 128, 0, 129, *refs) == 1    # channels > d
    assert lib.rkv_plan(0, 256, 128, 0, 0, *refs) == 1
    assert lib.rkv_plan(4096, 4, 128, 4, 0, *refs) == 1        # budget / 2 < page


def test_status_strings(lib):
    for code in range(6):
        assert lib.rkv_status_string(code)


FAKE = ctypes.c_void_p(1 << 20)   # aligned, non-null, never dereferenced: calls fail validation


def test_validation_rejects_before_launch(lib):
    vp = FAKE
    # hybrid: unsupported head_dim, gqa, bad page, odd budget, null pointer, small workspace
    common = (vp, None, None, vp, vp, vp, vp, vp)
    assert lib.rkv_hybrid_decode(*common, 1, 1, 4, 64, 64, 16, 256, 4, 32, 0.1, vp, None, None,
                                 None, vp, 256, None) == 2
    assert lib.rkv_hybrid_decode(*common, 1, 1, 3, 128, 64, 16, 256, 4, 32, 0.1, vp, None, None,
                                 None, vp, 256, None) == 2
    assert lib.rkv_hybrid_decode(*common, 1, 1, 4, 128, 64, 16, 256, 3, 32, 0.1, vp, None, None,
                                 None, vp, 256, None) == 1
    assert lib.rkv_hybrid_decode(*common, 1, 1, 4, 128, 64, 16, 255, 4, 32, 0.1, vp, None, None,
                                 None, vp, 256, None) == 1
    assert lib.rkv_hybrid_decode(*common, 1, 1, 4, 128, 64, 12, 256, 4, 32, 0.1, vp, None, None,
                                 None, vp, 256, None) == 1                      # page_cap % 8
    assert lib.rkv_hybrid_decode(None, None, None, vp, vp, vp, vp, vp, 1, 1, 4, 128, 64, 16, 256,
                                 4, 32, 0.1, vp, None, None, None, vp, 256, None) == 1
    assert lib.rkv_hybrid_decode(*common, 1, 1, 4, 128, 64, 16, 256, 4, 32, 0.1, vp, None, None,
                                 None, vp, 8, None) == 3
    # page_cap past the decode CTA's shared memory (190 KB: 31,168 pages at budget / page = 64)
    # is unsupported; at the limit the call gets as far as the workspace check (no workspace given)
    assert lib.rkv_hybrid_decode(*common, 1, 1, 4, 128, 64, 31176, 256, 4, 32, 0.1, vp, None,
                                 None, None, vp, 0, None) == 2
    assert lib.rkv_hybrid_decode(*common, 1, 1, 4, 128, 64, 31168, 256, 4, 32, 0.1, vp, None,
                                 None, None, vp, 0, None) == 3
    assert lib.rkv_hybrid_decode(vp, vp, None, vp, vp, vp, vp, vp, 1, 1, 4, 128, 64, 16, 256, 4,
                                 32, 0.1, vp, None, None, None, vp, 256, None) == 1  # new_v missing
    misaligned = ctypes.c_void_p((1 << 20) + 8)
    assert lib.rkv_hybrid_decode(misaligned, None, None, vp, vp, vp, vp, vp, 1, 1, 4, 128, 64, 16,
                                 256, 4, 32, 0.1, vp, None, None, None, vp, 256, None) == 1
    # dense
    assert lib.rkv_dense_decode(vp, vp, vp, vp, 1, 1, 4, 128, 100, 0.1, vp, vp, 16, None) == 3
    assert lib.rkv_dense_decode(vp, vp, vp, vp, 1, 1, 4, 128, 100, -1.0, vp, vp, 1 << 20,
                                None) == 1
    # summaries
    assert lib.rkv_build_page_summaries(vp, vp, 1, 1, 128, 64, 3, 16, 0, vp, vp, vp, 256,
                                        None) == 1
    assert lib.rkv_build_page_summaries(vp, vp, 1, 1, 128, 64, 4, 16, 0, vp, vp, vp, 4,
                                        None) == 3
    # snapkv: even kernel, keep <= window, gqa * window > 256, small workspace
    args = (vp, vp, vp, vp, 1, 2, 4, 128, 4096, 32)
    assert lib.rkv_snapkv_compress(*args, 6, 256, 0.1, vp, vp, 256, vp, vp, None, vp, 1 << 30,
                                   None) == 1
    assert lib.rkv_snapkv_compress(*args, 7, 32, 0.1, vp, vp, 256, vp, vp, None, vp, 1 << 30,
                                   None) == 1
    assert lib.rkv_snapkv_compress(*args, 7, 512, 0.1, vp, vp, 256, vp, vp, None, vp, 1 << 30,
                                   None) == 1                                  # keep > cap
    assert lib.rkv_snapkv_compress(vp, vp, vp, vp, 1, 2, 16, 128, 4096, 32, 7, 256, 0.1, vp, vp,
                                   256, vp, vp, None, vp, 1 << 30, None) == 2
    assert lib.rkv_snapkv_compress(*args, 7, 256, 0.1, vp, vp, 256, vp, vp, None, vp, 64,
                                   None) == 3



@pytest.mark.parametrize("ctx", [100, 4096, 8192, 30000, 32768, 65536, 131072, 1 << 20])
@pytest.mark.parametrize("budget", [64, 256, 512, 1024, 4096])
def test_plan_even_split_matches_oracle(lib, ctx, budget):
    from sparse_kv_cache_snapkv_gb300 import rkv
    assert rkv.rkv_plan_even_split(ctx, budget) == O.plan_even_split(ctx, budget, 128)


def test_per_head_compress_validation(lib):
    vp = FAKE
    args = (vp, vp, vp, vp, 1, 2, 4, 128, 4096, 32)
    big = 1 << 30
    # window over 256 rows, even kernel, keep <= window, gqa 0, small workspace
    assert lib.rkv_snapkv_compress_per_head(vp, vp, vp, vp, 1, 2, 4, 128, 4096, 300, 7, 512, 0.1,
                                            vp, vp, 512, vp, vp, None, vp, big, None) == 2
    assert lib.rkv_snapkv_compress_per_head(*args, 6, 256, 0.1, vp, vp, 256, vp, vp, None, vp,
                                            big, None) == 1
    assert lib.rkv_snapkv_compress_per_head(*args, 7, 32, 0.1, vp, vp, 256, vp, vp, None, vp,
                                            big, None) == 1
    assert lib.rkv_snapkv_compress_per_head(vp, vp, vp, vp, 1, 2, 0, 128, 4096, 32, 7, 256, 0.1,
                                            vp, vp, 256, vp, vp, None, vp, big, None) == 1
    assert lib.rkv_snapkv_compress_per_head(*args, 7, 256, 0.1, vp, vp, 256, vp, vp, None, vp, 64,
                                            None) == 3
    # the per-head workspace is the one of n_kv * gqa single-head units
    assert lib.rkv_snapkv_per_head_workspace_bytes(2, 8, 4, 32768, 32) == \
        lib.rkv_snapkv_workspace_bytes(2, 32, 1, 32768, 32)

def test_avg_pool_compress_validation(lib):
    vp = FAKE
    args = (vp, vp, vp, vp, 1, 2, 4, 128, 4096, 32)
    big = 1 << 30
    # even kernel, kernel past the fixed-point limit, keep <= window, small workspace
    assert lib.rkv_snapkv_compress_avg_pool(*args, 6, 256, 0.1, vp, vp, 256, vp, vp, None, vp,
                                            big, None) == 1
    assert lib.rkv_snapkv_compress_avg_pool(*args, (1 << 20) + 1, 256, 0.1, vp, vp, 256, vp, vp,
                                            None, vp, big, None) == 1
    assert lib.rkv_snapkv_compress_avg_pool(*args, 7, 32, 0.1, vp, vp, 256, vp, vp, None, vp,
                                            big, None) == 1
    assert lib.rkv_snapkv_compress_avg_pool(*args, 7, 256, 0.1, vp, vp, 256, vp, vp, None, vp, 64,
                                            None) == 3


def test_select_only_validation(lib):
    vp = FAKE
    big = 1 << 30
    # (k, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window, kernel, keep, scale)
    head = (vp, vp, vp, 1, 2, 4, 128, 4096, 32, 7)
    assert lib.rkv_snapkv_select(*head, 256, 0.1, vp, 255, vp, None, vp, big, None) == 1  # stride
    assert lib.rkv_snapkv_select(*head, 256, 0.1, vp, 0, vp, None, vp, big, None) == 1
    assert lib.rkv_snapkv_select(*head, 32, 0.1, vp, 512, vp, None, vp, big, None) == 1   # keep
    assert lib.rkv_snapkv_select(vp, vp, vp, 1, 2, 4, 64, 4096, 32, 7, 256, 0.1, vp, 256, vp,
                                 None, vp, big, None) == 2                              # head_dim
    assert lib.rkv_snapkv_select(*head, 256, 0.1, vp, 256, vp, None, vp, 64, None) == 3  # ws


def test_scores_only_validation(lib):
    vp = FAKE
    big = 1 << 30
    # (k, seq_lens, q_win, n, n_kv, gqa, head_dim, max_len, window, scale, scores_out, ws, ...)
    assert lib.rkv_snapkv_scores(vp, vp, vp, 1, 2, 4, 128, 4096, 32, 0.1, None, vp, big,
                                 None) == 1                                   # scores required
    assert lib.rkv_snapkv_scores(vp, vp, vp, 1, 2, 4, 128, 32, 32, 0.1, vp, vp, big,
                                 None) == 1                                   # max_len <= window
    assert lib.rkv_snapkv_scores(vp, vp, vp, 1, 2, 4, 128, 4096, 32, 0.0, vp, vp, big,
                                 None) == 1                                   # scale
    assert lib.rkv_snapkv_scores(vp, vp, vp, 1, 2, 4, 64, 4096, 32, 0.1, vp, vp, big,
                                 None) == 2                                   # head_dim
    assert lib.rkv_snapkv_scores(vp, vp, vp, 1, 2, 16, 128, 4096, 32, 0.1, vp, vp, big,
                                 None) == 2                                   # G * W > 256
    assert lib.rkv_snapkv_scores(vp, vp, vp, 1, 2, 4, 128, 4096, 32, 0.1, vp, vp, 64,
                                 None) == 3                                   # workspace


def test_wait_timeout_hook_validation(lib):
    vp = FAKE
    big = 1 << 30
    args = (vp, vp, vp, 1, 2, 4, 128, 4096, 32, 0.1, vp)
    assert lib.rkv_testing_scores_wait_timeout(*args, 10, vp, big, None) == 1        # too short
    assert lib.rkv_testing_scores_wait_timeout(*args, 2 * 10**9, vp, big, None) == 1  # too long
    assert lib.rkv_testing_scores_wait_timeout(*args, 10**6, vp, 64, None) == 3       # ws


def test_decode_layout_hook(lib):
    # include/rkv_testing.h: 0..2 accepted, anything else rejected; back to automatic after
    for bad in (-1, 3, 1 << 20):
        assert lib.rkv_testing_decode_layout(bad) == 1  # RKV_ERR_INVALID_ARG
    for ok in (1, 2, 0):
        assert lib.rkv_testing_decode_layout(ok) == 0


def test_mt_validation_rejects_before_launch(lib):
    vp = FAKE
    # (q, new_k, new_v, k_full, v_full, full_len, kept_idx, kept_len, kmin, kmax)
    ptrs = (vp, None, None, vp, vp, vp, vp, vp, vp, vp)
    tail = (0.1, vp, None, None, None, vp, 256, None)
    # n, n_kv, gqa, head_dim, full_cap, kcap, page_cap, budget, page, channels
    ok = (1, 1, 4, 128, 4096, 64, 16, 256, 4, 32)
    bad_cases = [
        ((1, 1, 4, 64, 4096, 64, 16, 256, 4, 32), 2),    # head_dim
        ((1, 1, 4, 128, 4096, 0, 16, 256, 4, 32), 1),    # kcap
        ((1, 1, 4, 128, 0, 64, 16, 256, 4, 32), 1),      # full_cap
        ((1, 1, 4, 128, 4096, 64, 12, 256, 4, 32), 1),   # page_cap % 8
        ((1, 1, 4, 128, 4096, 64, 16, 256, 4, 0), 1),    # channels
    ]
    for sizes, code in bad_cases:
        assert lib.rkv_hybrid_decode_mt(*ptrs, *sizes, *tail) == code, sizes
    no_kept = (vp, None, None, vp, vp, vp, None, vp, vp, vp)
    assert lib.rkv_hybrid_decode_mt(*no_kept, *ok, *tail) == 1
    no_full_len = (vp, None, None, vp, vp, None, vp, vp, vp, vp)
    assert lib.rkv_hybrid_decode_mt(*no_full_len, *ok, *tail) == 1
    assert lib.rkv_hybrid_decode_mt(*ptrs, *ok, 0.1, vp, None, None, None, vp, 8, None) == 3
    # summaries over a kept list: no list, bad page, small workspace
    assert lib.rkv_build_page_summaries_mt(vp, None, vp, 1, 1, 128, 4096, 64, 4, 16, 0, vp, vp,
                                           vp, 256, None) == 1
    assert lib.rkv_build_page_summaries_mt(vp, vp, vp, 1, 1, 128, 4096, 64, 3, 16, 0, vp, vp,
                                           vp, 256, None) == 1
    assert lib.rkv_build_page_summaries_mt(vp, vp, vp, 1, 1, 128, 4096, 64, 4, 16, 0, vp, vp,
                                           vp, 4, None) == 3


def test_workspace_sizes_monotone(lib):
    a = lib.rkv_dense_decode_workspace_bytes(32, 8, 4, 32768)
    b = lib.rkv_dense_decode_workspace_bytes(32, 8, 4, 131072)
    assert 256 < a <= b
    assert lib.rkv_snapkv_workspace_bytes(1, 8, 4, 131072, 64) > \
        lib.rkv_snapkv_workspace_bytes(1, 8, 4, 4096, 32)
    assert lib.rkv_hybrid_decode_workspace_bytes(32, 8, 4, 1024, 256, 4) >= 256


def test_binding_rejects_uneven_groups():
    from sparse_kv_cache_snapkv_gb300 import rkv
    with pytest.raises(ValueError):
        rkv._group(30, 8)
    assert rkv._group(32, 8) == 4
