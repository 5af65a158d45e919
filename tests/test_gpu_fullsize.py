"""Full-size parity in the launch configuration bench.py times: Llama-3.1-8B attention shapes,
32 layers x 8 KV heads, 32K prompt, budget 256 (keep 4096, page 4, 32 channels), run through the
same HotPath object; sampled (layer, KV head) units and decode steps are checked one by one
against the CPU oracle."""
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


def _check_units(hp, x, wl, samples, steps_to_check, seed):
    from sparse_kv_cache_snapkv_gb300 import rkv
    scale = hp.scale
    W = wl.window
    kernel = wl.kernel or O.adaptive_kernel_size(wl.max_len)
    S = (wl.budget // 2) // hp.page
    for (u, g) in samples:
        L = int(x["seq_lens"][u])
        k = _f64(x["k"][u, g, :L])
        v = _f64(x["v"][u, g, :L])
        q = _f64(x["q_win"][u, g * wl.gqa:(g + 1) * wl.gqa])
        score = O.window_scores(k, q, scale)
        pooled = O.pool_max(score, kernel)
        kept = hp.kept[u, g].cpu().numpy()
        n1 = int(hp.out_len[u])
        assert n1 == min(L, hp.keep)
        tag = f"unit {u} kv {g}"
        if L > hp.keep:
            assert np.array_equal(kept[hp.keep - W:], np.arange(L - W, L)), tag
            parity.check_selection(kept[:hp.keep - W], pooled, hp.keep - W, f"{tag} kept")
        kc = _f64(hp.k_out[u, g, :n1])
        vc = _f64(hp.v_out[u, g, :n1])
        assert np.array_equal(kc, k[kept[:n1]]) and np.array_equal(vc, v[kept[:n1]]), tag
        rmin, rmax = O.page_summaries(kc, n1, hp.page)
        P = rmin.shape[1]
        assert np.array_equal(_f64(hp.kmin[u, g, :, :P]), rmin), f"{tag} kmin"
        assert np.array_equal(_f64(hp.kmax[u, g, :, :P]), rmax), f"{tag} kmax"
    # decode steps re-run with the optional selection outputs (same kernel, same grid)
    for t in steps_to_check:
        sel = torch.empty(wl.n, wl.n_kv, S, dtype=torch.int32, device="cuda")
        out = torch.empty_like(hp.out[t])
        rkv.rkv_hybrid_decode(hp.dec_q[t], hp.k_out, hp.v_out, hp.length, hp.kmin, hp.kmax,
                              wl.budget, hp.page, hp.channels, scale, out, sel_pages=sel,
                              ws=hp.ws_dec)
        rkv.rkv_check_status(hp.ws_dec)
        assert torch.equal(out, hp.out[t]), "re-run differs from the timed launch"
        for (u, g) in samples:
            n1 = int(hp.out_len[u])
            kc = _f64(hp.k_out[u, g, :n1])
            vc = _f64(hp.v_out[u, g, :n1])
            rmin, rmax = O.page_summaries(kc, n1, hp.page)
            qh = _f64(hp.dec_q[t, u, g * wl.gqa:(g + 1) * wl.gqa])
            ref = O.hybrid_decode(qh, kc, vc, n1, rmin, rmax, wl.budget, hp.page, hp.channels,
                                  scale)
            tag = f"step {t} unit {u} kv {g}"
            gp = sel[u, g].cpu().numpy()
            if ref["pages"] is None:
                parity.check_attention(_f64(out[u, g * wl.gqa:(g + 1) * wl.gqa]), qh, kc[:n1],
                                       vc[:n1], scale, tag)
                continue
            parity.check_selection(gp, ref["scores"], len(ref["pages"]), tag)
            toks = np.concatenate([np.arange(p * hp.page, min(n1, (p + 1) * hp.page))
                                   for p in gp])
            parity.check_attention(_f64(out[u, g * wl.gqa:(g + 1) * wl.gqa]), qh, kc[toks],
                                   vc[toks], scale, tag)


def test_bench_workload_llama8b_32k():
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    from sparse_kv_cache_snapkv_gb300.pipeline import HotPath
    wl = S.WORKLOADS["llama8b_32k"]
    x = S.prefill_inputs(wl, seed=2000, device="cuda")
    dq = S.decode_queries(wl, wl.decode_steps, seed=2500, device="cuda")
    hp = HotPath(wl, x["k"], x["v"], x["q_win"], x["seq_lens"], dq)
    hp.step()
    torch.cuda.synchronize()
    hp.check_status()
    assert hp.keep == 4096 and hp.page == 4 and hp.channels == 32
    _check_units(hp, x, wl, [(0, 0), (15, 3), (31, 7)], [0, 64, 127], seed=1)
    del hp, x
    torch.cuda.empty_cache()
