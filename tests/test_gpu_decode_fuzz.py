"""Seeded random configurations of the hybrid decode (shapes, GQA ratio, budget, page, kept
channels, ragged lengths incl. dense ones), each checked against the oracle in both shared-memory
layouts; and seeded random runs of decode steps that append a token each (page boundaries,
lengths crossing the budget), checked step by step and by the final cache and summaries."""
import math

import numpy as np
import pytest
import torch

from oracle import rocketkv as O
from tests import parity
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


def _append_config(seed):
    r = np.random.default_rng(5000 + seed)
    gqa = int(r.choice([1, 2, 4, 8]))
    page = int(r.choice([1, 2, 4, 8, 16, 32, 64]))
    budget = 2 * page * int(r.integers(1, max(2, 512 // page)))
    channels = int(r.integers(1, 129))
    n, n_kv = int(r.integers(1, 4)), int(r.integers(1, 3))
    steps = int(r.integers(5, 25))
    lens = [int(x) for x in r.integers(1, 3000, size=n)]
    lens[0] = budget - int(r.integers(0, 3))   # crosses the dense boundary while appending
    lens[-1] = page * int(r.integers(1, 3000 // page + 1)) - 1   # one short of a page boundary
    lens = [max(1, L) for L in lens]
    return n, n_kv, gqa, lens, budget, page, channels, steps


@pytest.mark.parametrize("seed", range(16))
def test_decode_random_appends(seed):
    rkv = T._lib()
    n, n_kv, gqa, lens, B, page, C, steps = _append_config(seed)
    cap = max(lens) + steps + 1
    k, v = T._make_cache(n, n_kv, cap, lens, seed=6000 + seed)
    page_cap = T._page_cap(cap, page)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kmin, kmax = T._summaries(rkv, k, lens_t, page, page_cap)
    kk, vv = T._f64(k), T._f64(v)
    cur = list(lens)
    rmins, rmaxs = {}, {}
    for u in range(n):
        for g in range(n_kv):
            a, b = O.page_summaries(kk[u, g], cur[u], page)
            rmins[u, g] = np.zeros((T.D, page_cap))
            rmaxs[u, g] = np.zeros((T.D, page_cap))
            rmins[u, g][:, :a.shape[1]] = a
            rmaxs[u, g][:, :a.shape[1]] = b
    gen = torch.Generator().manual_seed(7000 + seed)
    scale = 1.0 / math.sqrt(T.D)
    S = (B // 2) // page
    for step in range(steps):
        q = torch.randn(n, n_kv * gqa, T.D, generator=gen).to(torch.bfloat16).cuda()
        nk = torch.randn(n, n_kv, T.D, generator=gen).to(torch.bfloat16).cuda()
        nv = torch.randn(n, n_kv, T.D, generator=gen).to(torch.bfloat16).cuda()
        out = torch.empty_like(q)
        sel_p = torch.empty(n, n_kv, S, dtype=torch.int32, device="cuda")
        ws = rkv.rkv_hybrid_decode(q, k, v, lens_t, kmin, kmax, B, page, C, scale, out,
                                   new_k=nk, new_v=nv, sel_pages=sel_p)
        rkv.rkv_check_status(ws)
        qq, nkk, nvv = T._f64(q), T._f64(nk), T._f64(nv)
        for u in range(n):
            for g in range(n_kv):
                newlen = O.append_token(kk[u, g], vv[u, g], cur[u], rmins[u, g], rmaxs[u, g],
                                        nkk[u, g], nvv[u, g], page)
            cur[u] = newlen
            for g in range(n_kv):
                qh = qq[u, g * gqa:(g + 1) * gqa]
                L = cur[u]
                ref = O.hybrid_decode(qh, kk[u, g], vv[u, g], L, rmins[u, g], rmaxs[u, g], B,
                                      page, C, scale)
                tag = f"seed {seed} step {step} unit {u} kv {g} len {L}"
                if ref["pages"] is None:
                    parity.check_attention(T._f64(out[u, g * gqa:(g + 1) * gqa]), qh,
                                           kk[u, g][:L], vv[u, g][:L], scale, tag)
                    continue
                gp = sel_p[u, g].cpu().numpy()
                parity.check_selection(gp, ref["scores"], len(ref["pages"]), tag)
                toks = np.concatenate([np.arange(pg * page, min(L, (pg + 1) * page))
                                       for pg in gp])
                parity.check_attention(T._f64(out[u, g * gqa:(g + 1) * gqa]), qh,
                                       kk[u, g][toks], vv[u, g][toks], scale, tag)
    assert lens_t.cpu().tolist() == cur
    for u in range(n):
        for g in range(n_kv):
            P = (cur[u] + page - 1) // page
            assert np.array_equal(T._f64(kmin[u, g, :, :P]), rmins[u, g][:, :P])
            assert np.array_equal(T._f64(kmax[u, g, :, :P]), rmaxs[u, g][:, :P])
            assert np.array_equal(T._f64(k[u, g, :cur[u]]), kk[u, g, :cur[u]])
            assert np.array_equal(T._f64(v[u, g, :cur[u]]), vv[u, g, :cur[u]])
