"""One small pass of the hot path on cuda:0, checked against the CPU oracle (used by smoke()):
a hybrid decode step over a small cache, and a SnapKV++ compression of a small prompt with the
page summaries of its compact cache."""
import math

import numpy as np
import torch

from oracle import rocketkv as O
from tests import parity


def run():
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    rkv.load()
    assert torch.cuda.is_available(), "smoke needs cuda:0"
    torch.cuda.set_device(0)
    n, n_kv, gqa, d, cap, page, budget, channels = 1, 2, 4, 128, 1024, 4, 256, 32
    L = 1021
    k, v = S.random_cache(n, n_kv, cap, d, seed=7)
    k, v = k.cuda(), v.cuda()
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    page_cap = cap // page
    kmin = torch.zeros(n, n_kv, d, page_cap, dtype=torch.bfloat16, device="cuda")
    kmax = torch.zeros_like(kmin)
    ws = rkv.rkv_build_page_summaries(k, lens, page, kmin, kmax)
    rkv.rkv_check_status(ws)
    q = torch.randn(n, n_kv * gqa, d, generator=torch.Generator().manual_seed(8))
    q = q.to(torch.bfloat16).cuda()
    out = torch.empty_like(q)
    sel = torch.empty(n, n_kv, budget // 2 // page, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    ws = rkv.rkv_hybrid_decode(q, k, v, lens, kmin, kmax, budget, page, channels, scale, out,
                               sel_pages=sel)
    rkv.rkv_check_status(ws)
    kk = k.double().cpu().numpy()
    vv = v.double().cpu().numpy()
    for g in range(n_kv):
        qh = q[0, g * gqa:(g + 1) * gqa].double().cpu().numpy()
        mn, mx = O.page_summaries(kk[0, g], L, page)
        ref = O.hybrid_decode(qh, kk[0, g], vv[0, g], L, mn, mx, budget, page, channels, scale)
        gp = sel[0, g].cpu().numpy()
        parity.check_selection(gp, ref["scores"], len(ref["pages"]), "smoke pages")
        toks = np.concatenate([np.arange(p * page, min(L, (p + 1) * page)) for p in gp])
        parity.check_attention(out[0, g * gqa:(g + 1) * gqa].double().cpu().numpy(), qh,
                               kk[0, g][toks], vv[0, g][toks], scale, "smoke out")
    # stage 1 on a small prompt: tensor-core window scores, pooling, top-k, gather with the page
    # summaries of the compact cache
    W, keep, kernel, Lp = 32, 1024, 7, 3001
    wl = S.Workload("smoke", 1, 1, n_kv, gqa, d, (Lp,), W, budget, needles=4)
    x = S.prefill_inputs(wl, seed=9, device="cuda")
    k_c = torch.zeros(1, n_kv, keep, d, dtype=torch.bfloat16, device="cuda")
    v_c = torch.zeros_like(k_c)
    kept = torch.empty(1, n_kv, keep, dtype=torch.int32, device="cuda")
    out_len = torch.empty(1, dtype=torch.int32, device="cuda")
    pc = ((keep + page - 1) // page + 7) // 8 * 8
    kmin_c = torch.zeros(1, n_kv, d, pc, dtype=torch.bfloat16, device="cuda")
    kmax_c = torch.zeros_like(kmin_c)
    scores = torch.empty(1, n_kv, Lp - W, dtype=torch.float32, device="cuda")
    ws = rkv.rkv_snapkv_compress_summarized(x["k"], x["v"], x["seq_lens"], x["q_win"], kernel,
                                            keep, scale, k_c, v_c, kept, out_len, page, kmin_c,
                                            kmax_c, scores_out=scores)
    rkv.rkv_check_status(ws)
    assert int(out_len[0]) == keep, "smoke compress length"
    for g in range(n_kv):
        kg = x["k"][0, g, :Lp].double().cpu().numpy()
        qw = x["q_win"][0, g * gqa:(g + 1) * gqa].double().cpu().numpy()
        ref = O.window_scores(kg, qw, scale)
        gs = scores[0, g].double().cpu().numpy()
        assert (np.abs(gs - ref) <= 1e-4 * np.abs(ref) + 1e-30).all(), "smoke scores"
        got = kept[0, g].cpu().numpy()
        assert np.array_equal(got[keep - W:], np.arange(Lp - W, Lp)), "smoke window"
        parity.check_selection(got[:keep - W], O.pool_max(ref, kernel), keep - W, "smoke kept")
        assert torch.equal(k_c[0, g], x["k"][0, g][kept[0, g].long()]), "smoke gather"
        mn, mx = O.page_summaries(k_c[0, g].double().cpu().numpy(), keep, page)
        P = mn.shape[1]
        assert np.array_equal(kmin_c[0, g, :, :P].double().cpu().numpy(), mn), "smoke kmin"
        assert np.array_equal(kmax_c[0, g, :, :P].double().cpu().numpy(), mx), "smoke kmax"
    print("smoke ok")
