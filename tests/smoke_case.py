"""One small pass of the hot path on cuda:0, checked against the CPU oracle (used by smoke())."""
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
        parity.check_output(out[0, g * gqa:(g + 1) * gqa].double().cpu().numpy(),
                            O.attention(qh, kk[0, g][toks], vv[0, g][toks], scale), "smoke out")
    print("smoke ok")
