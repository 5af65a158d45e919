"""Parity of the other workloads at (or near) their full sizes, on sampled units:

* 128K prompts, batch 4, budget 1024 (keep 16384), 4 outlier channels at 10x -- one layer;
* 16 ragged sequences of 8K..64K tokens, budget 512, decode with a new token appended per step;
* the 128K prefill sweep: window 64 (G * W = 256), pooling kernels {1,3,7,15,31} x budgets
  {256, 1024, 4096}.
"""
import math

import numpy as np
import pytest
import torch

from oracle import rocketkv as O
from tests import parity

pytestmark = pytest.mark.gpu

D = 128


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _check_compress(hp, x, wl, u, g, kernel, tag):
    L = int(x["seq_lens"][u])
    W = wl.window
    k = _f64(x["k"][u, g, :L])
    v = _f64(x["v"][u, g, :L])
    q = _f64(x["q_win"][u, g * wl.gqa:(g + 1) * wl.gqa])
    pooled = O.pool_max(O.window_scores(k, q, hp.scale), kernel)
    kept = hp.kept[u, g].cpu().numpy()
    n1 = int(hp.out_len[u])
    assert n1 == min(L, hp.keep), tag
    if L > hp.keep:
        assert np.array_equal(kept[hp.keep - W:], np.arange(L - W, L)), tag
        parity.check_selection(kept[:hp.keep - W], pooled, hp.keep - W, f"{tag} kept")
    kc, vc = k[kept[:n1]], v[kept[:n1]]
    assert np.array_equal(_f64(hp.k_out[u, g, :n1]), kc), tag
    assert np.array_equal(_f64(hp.v_out[u, g, :n1]), vc), tag
    return kc, vc


def _check_decode_step(rkv, hp, wl, t, samples, caches, new_tokens=False):
    S = (wl.budget // 2) // hp.page
    sel = torch.empty(wl.n, wl.n_kv, S, dtype=torch.int32, device="cuda")
    out = torch.empty_like(hp.out[t])
    nk = hp.new_k[t] if new_tokens else None
    nv = hp.new_v[t] if new_tokens else None
    rkv.rkv_hybrid_decode(hp.dec_q[t], hp.k_out, hp.v_out, hp.length, hp.kmin, hp.kmax,
                          wl.budget, hp.page, hp.channels, hp.scale, out, new_k=nk, new_v=nv,
                          sel_pages=sel, ws=hp.ws_dec)
    rkv.rkv_check_status(hp.ws_dec)
    for (u, g) in samples:
        st = caches[(u, g)]
        if new_tokens:
            st["len"] = O.append_token(st["k"], st["v"], st["len"], st["kmin"], st["kmax"],
                                       _f64(nk[u, g]), _f64(nv[u, g]), hp.page)
        L = st["len"]
        qh = _f64(hp.dec_q[t, u, g * wl.gqa:(g + 1) * wl.gqa])
        ref = O.hybrid_decode(qh, st["k"], st["v"], L, st["kmin"], st["kmax"], wl.budget,
                              hp.page, hp.channels, hp.scale)
        tag = f"step {t} unit {u} kv {g} len {L}"
        if ref["pages"] is None:
            parity.check_attention(_f64(out[u, g * wl.gqa:(g + 1) * wl.gqa]), qh, st["k"][:L],
                                   st["v"][:L], hp.scale, tag)
            continue
        gp = sel[u, g].cpu().numpy()
        parity.check_selection(gp, ref["scores"], len(ref["pages"]), tag)
        toks = np.concatenate([np.arange(p * hp.page, min(L, (p + 1) * hp.page)) for p in gp])
        parity.check_attention(_f64(out[u, g * wl.gqa:(g + 1) * wl.gqa]), qh, st["k"][toks],
                               st["v"][toks], hp.scale, tag)


def _cache_state(kc, vc, page, page_cap, cap):
    n1 = kc.shape[0]
    k = np.zeros((cap, D))
    v = np.zeros((cap, D))
    k[:n1], v[:n1] = kc, vc
    kmin = np.zeros((D, page_cap))
    kmax = np.zeros((D, page_cap))
    a, b = O.page_summaries(kc, n1, page)
    kmin[:, :a.shape[1]], kmax[:, :a.shape[1]] = a, b
    return {"k": k, "v": v, "kmin": kmin, "kmax": kmax, "len": n1}


def test_128k_batch4_budget1024_outliers():
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    from sparse_kv_cache_snapkv_gb300.pipeline import HotPath
    wl = S.WORKLOADS["llama8b_128k_b4"].with_layers(1)
    x = S.prefill_inputs(wl, seed=3000, device="cuda")
    dq = S.decode_queries(wl, 2, seed=3500, device="cuda")
    hp = HotPath(wl, x["k"], x["v"], x["q_win"], x["seq_lens"], dq)
    assert hp.keep == 16384
    hp.compress()
    hp.summaries()
    torch.cuda.synchronize()
    hp.check_status()
    samples = [(0, 0), (3, 5)]
    caches = {}
    for (u, g) in samples:
        kc, vc = _check_compress(hp, x, wl, u, g, 31, f"128k unit {u} kv {g}")
        caches[(u, g)] = _cache_state(kc, vc, hp.page, hp.page_cap, hp.cap)
        P = (kc.shape[0] + hp.page - 1) // hp.page
        assert np.array_equal(_f64(hp.kmin[u, g, :, :P]), caches[(u, g)]["kmin"][:, :P])
        assert np.array_equal(_f64(hp.kmax[u, g, :, :P]), caches[(u, g)]["kmax"][:, :P])
    rkv.load()
    for t in range(2):
        _check_decode_step(rkv, hp, wl, t, samples, caches)
    del hp, x
    torch.cuda.empty_cache()


def test_ragged16_budget512_with_appends():
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    from sparse_kv_cache_snapkv_gb300.pipeline import HotPath
    wl = S.WORKLOADS["ragged16"]
    steps = 24
    x = S.prefill_inputs(wl, seed=4000, device="cuda")
    dq = S.decode_queries(wl, steps, seed=4500, device="cuda")
    nk, nv = S.append_tokens(wl, steps, x["sigma"], seed=4900, device="cuda")
    hp = HotPath(wl, x["k"], x["v"], x["q_win"], x["seq_lens"], dq, nk, nv)
    assert hp.keep == 8192
    hp.compress()
    hp.summaries()
    torch.cuda.synchronize()
    hp.check_status()
    lens = x["seq_lens"].cpu().tolist()
    shortest = int(np.argmin(lens))
    longest = int(np.argmax(lens))
    samples = [(shortest, 0), (longest, 7), (5, 3)]
    caches = {}
    for (u, g) in samples:
        kernel = O.adaptive_kernel_size(lens[u])
        kc, vc = _check_compress(hp, x, wl, u, g, kernel, f"ragged unit {u} kv {g}")
        caches[(u, g)] = _cache_state(kc, vc, hp.page, hp.page_cap, hp.cap)
    rkv.load()
    for t in range(steps):
        _check_decode_step(rkv, hp, wl, t, samples, caches, new_tokens=True)
    assert hp.length.cpu().tolist() == [min(L, hp.keep) + steps for L in lens]
    for (u, g) in samples:
        st = caches[(u, g)]
        P = (st["len"] + hp.page - 1) // hp.page
        assert np.array_equal(_f64(hp.kmin[u, g, :, :P]), st["kmin"][:, :P])
        assert np.array_equal(_f64(hp.kmax[u, g, :, :P]), st["kmax"][:, :P])
    del hp, x
    torch.cuda.empty_cache()


def test_prefill_128k_window64_kernel_and_budget_sweep():
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    wl = S.WORKLOADS["prefill128k"]
    x = S.prefill_inputs(wl, seed=5000, device="cuda")
    rkv.load()
    n, n_kv, max_len = wl.n, wl.n_kv, wl.max_len
    W = wl.window
    scale = 1.0 / math.sqrt(D)
    samples = [0, 6]
    ref_scores = {}
    for g in samples:
        k = _f64(x["k"][0, g])
        q = _f64(x["q_win"][0, g * wl.gqa:(g + 1) * wl.gqa])
        ref_scores[g] = O.window_scores(k, q, scale)
    for budget in (256, 1024, 4096):
        keep = rkv.rkv_plan(max_len, budget)[0]
        k_out = torch.zeros(n, n_kv, keep, D, dtype=torch.bfloat16, device="cuda")
        v_out = torch.zeros_like(k_out)
        kept = torch.empty(n, n_kv, keep, dtype=torch.int32, device="cuda")
        out_len = torch.empty(n, dtype=torch.int32, device="cuda")
        scores = torch.empty(n, n_kv, max_len - W, dtype=torch.float32, device="cuda")
        for kernel in (1, 3, 7, 15, 31):
            ws = rkv.rkv_snapkv_compress(x["k"], x["v"], x["seq_lens"], x["q_win"], kernel, keep,
                                         scale, k_out, v_out, kept, out_len, scores_out=scores)
            rkv.rkv_check_status(ws)
            for g in samples:
                tag = f"budget {budget} kernel {kernel} kv {g}"
                gs = scores[0, g].cpu().numpy().astype(np.float64)
                ref = ref_scores[g]
                assert (np.abs(gs - ref) <= 1e-4 * np.abs(ref) + 1e-30).all(), tag
                pooled = O.pool_max(ref, kernel)
                got = kept[0, g].cpu().numpy()
                assert np.array_equal(got[keep - W:], np.arange(max_len - W, max_len)), tag
                parity.check_selection(got[:keep - W], pooled, keep - W, tag)
                assert torch.equal(k_out[0, g], x["k"][0, g][kept[0, g].long()]), tag
    del x
    torch.cuda.empty_cache()
