"""The allocation-free dense decode (rkv_dense_decode_noalloc) against the workspace version.

Callers such as a plugin that is handed only its input and output tensors, or a host whose device
memory all belongs to its own pool, cannot call cudaMalloc for a workspace; this entry point keeps its scratch in a
fixed device array inside the library instead. The test calls it twice in a row through the C
ABI (different queries each time, so nothing may leak from the first call into the second) and
checks each output against rkv_dense_decode's bit for bit: both run the same kernels with the
same split plan, so nothing but the scratch location differs. It is collected last so that a
run stopping at the first failure has run the others.
"""
import numpy as np
import pytest
import torch


pytestmark = pytest.mark.gpu

D = 128


def test_dense_decode_noalloc_matches_workspace_version():
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    rkv.load()
    n, n_kv, gqa, max_len = 3, 2, 4, 5000
    lens = [5000, 1, 2049]
    k, v = S.random_cache(n, n_kv, max_len, D, seed=81)
    for u, L in enumerate(lens):
        k[u, :, L:] = 0
        v[u, :, L:] = 0
    k, v = k.cuda(), v.cuda()
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    gen = torch.Generator().manual_seed(82)
    for call in range(2):
        q = torch.randn(n, n_kv * gqa, D, generator=gen).to(torch.bfloat16).cuda()
        ref = torch.empty_like(q)
        ws = rkv.rkv_dense_decode(q, k, v, lens_t, 0.0884, ref)
        rkv.rkv_check_status(ws)
        out = torch.full_like(q, float("nan"))
        rkv.rkv_dense_decode_noalloc(q, k, v, lens_t, 0.0884, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"no-alloc call {call} differs from the workspace call"


def test_dense_decode_noalloc_rejects_oversize():
    from sparse_kv_cache_snapkv_gb300 import rkv
    lib = rkv.load()
    # 512 units x 64 query heads: the split partials alone need 16 MiB, beyond the fixed 8 MiB.
    # The size is checked before the pointers, so null pointers still get the size check's
    # answer (and nothing could be launched on them if the order of the checks ever changed).
    assert lib.rkv_dense_decode_workspace_bytes(512, 8, 8, 1024) > (8 << 20)
    code = lib.rkv_dense_decode_noalloc(None, None, None, None, 512, 8, 8, 128, 1024, 0.1,
                                        None, None)
    assert code == 6
    assert "too large" in rkv.rkv_status_string(6)
