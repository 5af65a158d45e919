"""Parity of the stage-2 kernels (page summaries, hybrid decode, append, dense decode) against
the CPU oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

from oracle import rocketkv as O
from tests import parity

pytestmark = pytest.mark.gpu

D = 128


def _lib():
    from sparse_kv_cache_snapkv_gb300 import rkv
    rkv.load()
    return rkv


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _page_cap(cap, page):
    return ((cap + page - 1) // page + 7) // 8 * 8


def _make_cache(n, n_kv, cap, lens, seed):
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    k, v = S.random_cache(n, n_kv, cap, D, seed)
    for u, L in enumerate(lens):
        k[u, :, L:] = 0
        v[u, :, L:] = 0
    return k.cuda(), v.cuda()


def _summaries(rkv, k, lens_t, page, page_cap):
    n, n_kv = k.shape[:2]
    kmin = torch.zeros(n, n_kv, D, page_cap, dtype=torch.bfloat16, device="cuda")
    kmax = torch.zeros_like(kmin)
    ws = rkv.rkv_build_page_summaries(k, lens_t, page, kmin, kmax)
    rkv.rkv_check_status(ws)
    return kmin, kmax


@pytest.mark.parametrize("page", [1, 4, 16])
def test_summaries_bit_exact(page):
    rkv = _lib()
    lens = [4093, 257, 1030]
    cap = 4096
    k, _ = _make_cache(3, 2, cap, lens, seed=11 + page)
    page_cap = _page_cap(cap, page)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kmin, kmax = _summaries(rkv, k, lens_t, page, page_cap)
    for u, L in enumerate(lens):
        for g in range(2):
            rmin, rmax = O.page_summaries(_f64(k[u, g]), L, page)
            P = rmin.shape[1]
            assert np.array_equal(_f64(kmin[u, g, :, :P]), rmin)
            assert np.array_equal(_f64(kmax[u, g, :, :P]), rmax)


def test_summaries_incremental_first_token():
    rkv = _lib()
    cap, page = 2048, 4
    lens = [1999, 2048]
    k, _ = _make_cache(2, 2, cap, lens, seed=5)
    page_cap = _page_cap(cap, page)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kmin, kmax = _summaries(rkv, k, lens_t, page, page_cap)
    full_min, full_max = kmin.clone(), kmax.clone()
    # scribble over the tail pages, then rebuild only from token 1500 on
    kmin[..., 375:] = 0
    kmax[..., 375:] = 0
    ws = rkv.rkv_build_page_summaries(k, lens_t, page, kmin, kmax, first_token=1500)
    rkv.rkv_check_status(ws)
    for u, L in enumerate(lens):
        P = (L + page - 1) // page
        assert torch.equal(kmin[u, :, :, :P], full_min[u, :, :, :P])
        assert torch.equal(kmax[u, :, :, :P], full_max[u, :, :, :P])


def _hybrid_case(n, n_kv, gqa, lens, cap, budget, page, channels, seed, steps=2, tweak=None):
    rkv = _lib()
    k, v = _make_cache(n, n_kv, cap, lens, seed)
    if tweak is not None:
        tweak(k, v)
    page_cap = _page_cap(cap, page)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kmin, kmax = _summaries(rkv, k, lens_t, page, page_cap)
    scale = 1.0 / math.sqrt(D)
    S = (budget // 2) // page
    g_ = torch.Generator().manual_seed(seed + 1)
    kk, vv = _f64(k), _f64(v)
    for step in range(steps):
        q = torch.randn(n, n_kv * gqa, D, generator=g_).to(torch.bfloat16).cuda()
        out = torch.empty_like(q)
        sel_c = torch.full((n, n_kv, channels), -7, dtype=torch.int32, device="cuda")
        sel_p = torch.full((n, n_kv, S), -7, dtype=torch.int32, device="cuda")
        approx = torch.zeros(n, n_kv, page_cap, dtype=torch.float32, device="cuda")
        ws = rkv.rkv_hybrid_decode(q, k, v, lens_t, kmin, kmax, budget, page, channels, scale,
                                   out, sel_channels=sel_c, sel_pages=sel_p,
                                   approx_scores=approx)
        rkv.rkv_check_status(ws)
        qq = _f64(q)
        for u, L in enumerate(lens):
            for g in range(n_kv):
                qh = qq[u, g * gqa:(g + 1) * gqa]
                rmin, rmax = O.page_summaries(kk[u, g], L, page)
                ref = O.hybrid_decode(qh, kk[u, g], vv[u, g], L, rmin, rmax, budget, page,
                                      channels, scale)
                tag = f"step {step} unit {u} kv {g} len {L}"
                if ref["channels"] is None:
                    assert (sel_c[u, g] == -1).all(), tag
                    assert (sel_p[u, g] == -1).all(), tag
                    parity.check_attention(_f64(out[u, g * gqa:(g + 1) * gqa]), qh, kk[u, g][:L],
                                           vv[u, g][:L], scale, tag)
                    continue
                mag = np.abs(qh).sum(axis=0)
                parity.check_selection(sel_c[u, g].cpu().numpy(), mag, channels,
                                       f"{tag} channels")
                gch = np.sort(sel_c[u, g].cpu().numpy())
                q_g = qh.sum(axis=0)
                # approximate scores: recompute on the GPU's channels (equal unless tie band)
                ref_a = O.approx_scores(q_g, gch, rmin, rmax)
                P = rmin.shape[1]
                magn = parity.approx_magnitude(q_g, gch, rmin, rmax)
                parity.check_approx(approx[u, g, :P].cpu().numpy(), ref_a, magn, len(gch),
                                    f"{tag} approx")
                nsel = min(S, P)
                gp = sel_p[u, g].cpu().numpy()
                assert (gp[nsel:] == -1).all(), tag
                parity.check_selection(gp[:nsel], ref_a, nsel, f"{tag} pages")
                assert np.all(np.diff(gp[:nsel]) > 0), f"{tag} pages not ascending"
                toks = np.concatenate([np.arange(pg * page, min(L, (pg + 1) * page))
                                       for pg in gp[:nsel]])
                parity.check_attention(_f64(out[u, g * gqa:(g + 1) * gqa]), qh, kk[u, g][toks],
                                       vv[u, g][toks], scale, tag)


def test_hybrid_config1_shape():
    # 8 q / 2 kv heads, 4K cache, B 256, page 4, 32 channels (the tiny configuration's decode)
    _hybrid_case(1, 2, 4, [4096], 4096, 256, 4, 32, seed=21, steps=4)


def test_hybrid_ragged_and_dense_fallback():
    # ragged lengths incl. a partial last page, P % 8 != 0, and len <= budget (dense path)
    _hybrid_case(4, 2, 4, [4093, 200, 1030, 256], 4096, 256, 4, 32, seed=22)


@pytest.mark.parametrize("gqa", [1, 2, 8])
def test_hybrid_gqa_variants(gqa):
    _hybrid_case(2, 2, gqa, [3001, 777], 3072, 256, 4, 32, seed=23 + gqa)


@pytest.mark.parametrize("budget,page,channels", [(1024, 4, 32), (256, 16, 128), (128, 1, 16),
                                                  (512, 8, 64)])
def test_hybrid_budget_page_channel_variants(budget, page, channels):
    _hybrid_case(2, 2, 4, [8191, 5000], 8192, budget, page, channels, seed=31 + page)


def test_hybrid_more_than_4096_pages_general_select():
    # 20,001 cached tokens in pages of 4 (5001 pages): the page select takes the general block
    # select instead of the register-resident one (<= 4096 pages); a second unit stays below it
    _hybrid_case(2, 1, 4, [20001, 3000], 20480, 512, 4, 32, seed=41, steps=1)


def test_hybrid_page1_all_channels_is_exact_group_topk():
    # the reduction the method's approximation collapses to (exact group top-k attention)
    rkv = _lib()
    n, n_kv, gqa, L, B = 1, 2, 4, 2000, 256
    k, v = _make_cache(n, n_kv, 2048, [L], seed=41)
    lens_t = torch.tensor([L], dtype=torch.int32, device="cuda")
    page_cap = _page_cap(2048, 1)
    kmin, kmax = _summaries(rkv, k, lens_t, 1, page_cap)
    q = torch.randn(n, n_kv * gqa, D, generator=torch.Generator().manual_seed(42))
    q = q.to(torch.bfloat16).cuda()
    out = torch.empty_like(q)
    sel_p = torch.empty(n, n_kv, B // 2, dtype=torch.int32, device="cuda")
    ws = rkv.rkv_hybrid_decode(q, k, v, lens_t, kmin, kmax, B, 1, D, 0.1, out, sel_pages=sel_p)
    rkv.rkv_check_status(ws)
    for g in range(n_kv):
        qh = _f64(q[0, g * gqa:(g + 1) * gqa])
        ref_out, ref_tok = O.group_topk_attention(qh, _f64(k[0, g]), _f64(v[0, g]), L, B // 2,
                                                  0.1)
        true = _f64(k[0, g])[:L] @ qh.sum(axis=0)
        parity.check_selection(sel_p[0, g].cpu().numpy(), true, B // 2, "exact top-k")
        toks = np.sort(np.asarray(ref_tok, dtype=np.int64))
        parity.check_attention(_f64(out[0, g * gqa:(g + 1) * gqa]), qh, _f64(k[0, g])[toks],
                               _f64(v[0, g])[toks], 0.1, "exact top-k out")
        assert np.allclose(O.attention(qh, _f64(k[0, g])[toks], _f64(v[0, g])[toks], 0.1),
                           ref_out, rtol=1e-12, atol=1e-12), "group_topk_attention's tokens"


def test_hybrid_append_steps():
    rkv = _lib()
    n, n_kv, gqa, page, B, C = 3, 2, 4, 4, 256, 32
    cap = 1100
    lens = [1021, 400, 200]          # 200 crosses the budget while appending
    k, v = _make_cache(n, n_kv, cap, lens, seed=51)
    page_cap = _page_cap(cap, page)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kmin, kmax = _summaries(rkv, k, lens_t, page, page_cap)
    kk, vv = _f64(k), _f64(v)
    cur = list(lens)
    rmins, rmaxs = {}, {}
    for u in range(n):
        for g in range(n_kv):
            a, b = O.page_summaries(kk[u, g], cur[u], page)
            rmins[u, g] = np.zeros((D, page_cap))
            rmaxs[u, g] = np.zeros((D, page_cap))
            rmins[u, g][:, :a.shape[1]] = a
            rmaxs[u, g][:, :a.shape[1]] = b
    gen = torch.Generator().manual_seed(52)
    scale = 1.0 / math.sqrt(D)
    for step in range(70):
        q = torch.randn(n, n_kv * gqa, D, generator=gen).to(torch.bfloat16).cuda()
        nk = torch.randn(n, n_kv, D, generator=gen).to(torch.bfloat16).cuda()
        nv = torch.randn(n, n_kv, D, generator=gen).to(torch.bfloat16).cuda()
        out = torch.empty_like(q)
        sel_p = torch.empty(n, n_kv, B // 2 // page, dtype=torch.int32, device="cuda")
        ws = rkv.rkv_hybrid_decode(q, k, v, lens_t, kmin, kmax, B, page, C, scale, out,
                                   new_k=nk, new_v=nv, sel_pages=sel_p)
        rkv.rkv_check_status(ws)
        qq, nkk, nvv = _f64(q), _f64(nk), _f64(nv)
        for u in range(n):
            newlen = None
            for g in range(n_kv):
                newlen = O.append_token(kk[u, g], vv[u, g], cur[u], rmins[u, g], rmaxs[u, g],
                                        nkk[u, g], nvv[u, g], page)
            cur[u] = newlen
            for g in range(n_kv):
                qh = qq[u, g * gqa:(g + 1) * gqa]
                L = cur[u]
                ref = O.hybrid_decode(qh, kk[u, g], vv[u, g], L, rmins[u, g], rmaxs[u, g], B,
                                      page, C, scale)
                tag = f"append step {step} unit {u} kv {g} len {L}"
                if ref["pages"] is None:
                    parity.check_attention(_f64(out[u, g * gqa:(g + 1) * gqa]), qh,
                                           kk[u, g][:L], vv[u, g][:L], scale, tag)
                    continue
                gp = sel_p[u, g].cpu().numpy()
                parity.check_selection(gp, ref["scores"], len(ref["pages"]), tag)
                toks = np.concatenate([np.arange(pg * page, min(L, (pg + 1) * page))
                                       for pg in gp])
                parity.check_attention(_f64(out[u, g * gqa:(g + 1) * gqa]), qh, kk[u, g][toks],
                                       vv[u, g][toks], scale, tag)
    assert lens_t.cpu().tolist() == cur
    for u in range(n):
        for g in range(n_kv):
            P = (cur[u] + page - 1) // page
            assert np.array_equal(_f64(kmin[u, g, :, :P]), rmins[u, g][:, :P])
            assert np.array_equal(_f64(kmax[u, g, :, :P]), rmaxs[u, g][:, :P])
            assert np.array_equal(_f64(k[u, g, :cur[u]]), kk[u, g, :cur[u]])


@pytest.mark.parametrize("gqa", [1, 4, 8])
def test_dense_decode_ragged(gqa):
    rkv = _lib()
    n, n_kv, max_len = 3, 2, 5000
    lens = [5000, 1, 2049]
    k, v = _make_cache(n, n_kv, max_len, lens, seed=61)
    q = torch.randn(n, n_kv * gqa, D, generator=torch.Generator().manual_seed(62))
    q = q.to(torch.bfloat16).cuda()
    out = torch.empty_like(q)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = rkv.rkv_dense_decode(q, k, v, lens_t, 0.0884, out)
    rkv.rkv_check_status(ws)
    kk, vv, qq = _f64(k), _f64(v), _f64(q)
    for u, L in enumerate(lens):
        for g in range(n_kv):
            qh = qq[u, g * gqa:(g + 1) * gqa]
            parity.check_attention(_f64(out[u, g * gqa:(g + 1) * gqa]), qh, kk[u, g][:L],
                                   vv[u, g][:L], 0.0884, f"dense {u} {g}")


def test_device_status_len_over_cap():
    rkv = _lib()
    k, v = _make_cache(1, 1, 64, [64], seed=71)
    lens_t = torch.tensor([65], dtype=torch.int32, device="cuda")   # beyond cap
    kmin = torch.zeros(1, 1, D, 16, dtype=torch.bfloat16, device="cuda")
    kmax = torch.zeros_like(kmin)
    ws = rkv.rkv_build_page_summaries(k, lens_t, 4, kmin, kmax)
    with pytest.raises(rkv.RkvError) as ei:
        rkv.rkv_check_status(ws)
    assert ei.value.bits & 1
    # the word is cleared by the check
    assert rkv.rkv_check_status(ws) == 0


def test_hybrid_page_select_heavy_tail():
    # a few pages whose keys are 300x larger (both signs): a score range dominated by outliers,
    # with the k-th page among the crowded ordinary ones
    def tweak(k, v):
        k[:, :, 40:52] *= 300
        k[:, :, 2000:2004] *= -300
    _hybrid_case(2, 2, 4, [4096, 3001], 4096, 256, 4, 32, seed=61, steps=3, tweak=tweak)


def test_hybrid_page_select_crowded_equal_scores():
    # 1004 identical pages (equal approximate scores) and 20 pages with 4x larger keys: the
    # k-th page lies among a thousand equal scores, which the select resolves down to the last
    # bit; the equal pages are then taken lowest index first, checked exactly on the kernel's
    # own scores
    rkv = _lib()
    n, n_kv, gqa, L, B, page, C = 1, 2, 4, 4096, 256, 4, 32
    k, v = _make_cache(n, n_kv, L, [L], seed=63)
    row = k[:, :, 0:1].clone()
    k[:, :, :] = row.expand(-1, -1, L, -1)
    k[:, :, 4000:4080] = row.expand(-1, -1, 80, -1) * 4
    lens_t = torch.tensor([L], dtype=torch.int32, device="cuda")
    page_cap = _page_cap(L, page)
    kmin, kmax = _summaries(rkv, k, lens_t, page, page_cap)
    S = B // 2 // page
    q = row[:, :, 0].repeat_interleave(gqa, dim=1).float()
    q = (q + 0.01 * torch.randn(q.shape, generator=torch.Generator().manual_seed(64)).cuda())
    q = q.to(torch.bfloat16)
    out = torch.empty_like(q)
    sel_c = torch.empty(n, n_kv, C, dtype=torch.int32, device="cuda")
    sel_p = torch.empty(n, n_kv, S, dtype=torch.int32, device="cuda")
    approx = torch.zeros(n, n_kv, page_cap, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    ws = rkv.rkv_hybrid_decode(q, k, v, lens_t, kmin, kmax, B, page, C, scale, out,
                               sel_channels=sel_c, sel_pages=sel_p, approx_scores=approx)
    rkv.rkv_check_status(ws)
    kk, vv, qq = _f64(k), _f64(v), _f64(q)
    P = L // page
    for g in range(n_kv):
        a = approx[0, g, :P].cpu().numpy().astype(np.float64)
        order = np.lexsort((np.arange(P), -a))
        gp = sel_p[0, g].cpu().numpy()
        assert np.array_equal(gp, np.sort(order[:S])), f"kv {g}: exact rule on own scores"
        # the k-th score is shared by hundreds of pages
        assert (a == a[order[S - 1]]).sum() > 1000, f"kv {g}: case not crowded"
        # and the selection is the oracle's within the tie band
        qh = qq[0, g * gqa:(g + 1) * gqa]
        rmin, rmax = O.page_summaries(kk[0, g], L, page)
        gch = np.sort(sel_c[0, g].cpu().numpy())
        ref_a = O.approx_scores(qh.sum(axis=0), gch, rmin, rmax)
        parity.check_selection(gp, ref_a, S, f"kv {g} pages")
        toks = np.concatenate([np.arange(pg * page, (pg + 1) * page) for pg in gp])
        parity.check_attention(_f64(out[0, g * gqa:(g + 1) * gqa]), qh, kk[0, g][toks],
                               vv[0, g][toks], scale, f"kv {g}")


def test_hybrid_exact_ties_take_lowest_pages_and_channels():
    # identical keys -> every page scores the same; a query whose |q| is equal on every channel
    # -> every channel ties. Both selections must then be the lowest indices.
    rkv = _lib()
    n, n_kv, gqa, L, B, page, C = 1, 1, 4, 1000, 256, 4, 32
    row = torch.randn(D, generator=torch.Generator().manual_seed(91)).to(torch.bfloat16)
    k = row.expand(n, n_kv, 1024, D).contiguous().cuda()
    v = torch.randn(n, n_kv, 1024, D, generator=torch.Generator().manual_seed(92))
    v = v.to(torch.bfloat16).cuda()
    lens_t = torch.tensor([L], dtype=torch.int32, device="cuda")
    kmin, kmax = _summaries(rkv, k, lens_t, page, 256)
    q = torch.ones(n, n_kv * gqa, D, dtype=torch.bfloat16, device="cuda")
    q[:, :, 1::2] = -1.0
    out = torch.empty_like(q)
    sel_c = torch.empty(n, n_kv, C, dtype=torch.int32, device="cuda")
    sel_p = torch.empty(n, n_kv, B // 2 // page, dtype=torch.int32, device="cuda")
    ws = rkv.rkv_hybrid_decode(q, k, v, lens_t, kmin, kmax, B, page, C, 0.1, out,
                               sel_channels=sel_c, sel_pages=sel_p)
    rkv.rkv_check_status(ws)
    assert sel_c[0, 0].tolist() == list(range(C))
    assert sel_p[0, 0].tolist() == list(range(B // 2 // page))
    parity.check_attention(_f64(out[0]), _f64(q[0]), _f64(k[0, 0, :128]), _f64(v[0, 0, :128]),
                           0.1, "all-ties output")
