"""RocketKV-MT through the C ABI: the full cache stays, the decode reads the kept tokens through
the index list stage 1 wrote.

The MT calls must compute exactly what the compact-cache calls compute on the gathered rows (the
same values in the same order), so their summaries, selections and outputs are compared with the
compact path bit for bit, with and without decode-time appends; a sample is also checked against
the oracle's MT functions, and a kept index out of range must raise the device status bit.
"""
import math

import numpy as np
import pytest
import torch

from oracle import rocketkv as O
from tests import parity

pytestmark = pytest.mark.gpu

D = 128
W = 32
BUDGET = 256
PAGE = 4
CHANNELS = 32


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _setup(lens, steps, seed):
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    rkv.load()
    wl = S.Workload("mt", len(lens), 1, 2, 4, D, tuple(lens), W, BUDGET, needles=8)
    x = S.prefill_inputs(wl, seed=seed, device="cuda")
    n, n_kv, max_len = wl.n, wl.n_kv, wl.max_len
    keep = rkv.rkv_plan(max_len, BUDGET)[0]
    kcap = keep + steps
    page_cap = ((kcap + PAGE - 1) // PAGE + 7) // 8 * 8
    scale = 1.0 / math.sqrt(D)
    # stage 1 into a compact cache with room for the appends
    k_c = torch.zeros(n, n_kv, kcap, D, dtype=torch.bfloat16, device="cuda")
    v_c = torch.zeros_like(k_c)
    kept = torch.empty(n, n_kv, keep, dtype=torch.int32, device="cuda")
    out_len = torch.empty(n, dtype=torch.int32, device="cuda")
    ws = rkv.rkv_snapkv_compress(x["k"], x["v"], x["seq_lens"], x["q_win"], 0, keep, scale, k_c,
                                 v_c, kept, out_len)
    rkv.rkv_check_status(ws)
    # MT state: the full cache (with room for the appends) and the kept list
    full_cap = max_len + steps
    k_f = torch.zeros(n, n_kv, full_cap, D, dtype=torch.bfloat16, device="cuda")
    v_f = torch.zeros_like(k_f)
    k_f[:, :, :max_len] = x["k"]
    v_f[:, :, :max_len] = x["v"]
    kept_mt = torch.full((n, n_kv, kcap), -1, dtype=torch.int32, device="cuda")
    kept_mt[:, :, :keep] = kept
    st = {"rkv": rkv, "x": x, "wl": wl, "scale": scale, "keep": keep, "kcap": kcap,
          "page_cap": page_cap, "k_c": k_c, "v_c": v_c, "len_c": out_len.clone(), "k_f": k_f,
          "v_f": v_f, "full_len": x["seq_lens"].clone(), "kept": kept_mt,
          "kept_len": out_len.clone()}
    z = lambda: torch.zeros(n, n_kv, D, page_cap, dtype=torch.bfloat16, device="cuda")
    st["kmin_c"], st["kmax_c"], st["kmin_m"], st["kmax_m"] = z(), z(), z(), z()
    rkv.rkv_check_status(rkv.rkv_build_page_summaries(k_c, st["len_c"], PAGE, st["kmin_c"],
                                                      st["kmax_c"]))
    rkv.rkv_check_status(rkv.rkv_build_page_summaries_mt(k_f, kept_mt, st["kept_len"], PAGE,
                                                         st["kmin_m"], st["kmax_m"]))
    return st


def _step(st, q, new_k=None, new_v=None):
    rkv = st["rkv"]
    n, n_kv = st["wl"].n, st["wl"].n_kv
    S_pages = (BUDGET // 2) // PAGE
    res = {}
    for mode in ("c", "m"):
        out = torch.empty_like(q)
        selp = torch.empty(n, n_kv, S_pages, dtype=torch.int32, device="cuda")
        selc = torch.empty(n, n_kv, CHANNELS, dtype=torch.int32, device="cuda")
        if mode == "c":
            ws = rkv.rkv_hybrid_decode(q, st["k_c"], st["v_c"], st["len_c"], st["kmin_c"],
                                       st["kmax_c"], BUDGET, PAGE, CHANNELS, st["scale"], out,
                                       new_k=new_k, new_v=new_v, sel_channels=selc,
                                       sel_pages=selp)
        else:
            ws = rkv.rkv_hybrid_decode_mt(q, st["k_f"], st["v_f"], st["full_len"], st["kept"],
                                          st["kept_len"], st["kmin_m"], st["kmax_m"], BUDGET,
                                          PAGE, CHANNELS, st["scale"], out, new_k=new_k,
                                          new_v=new_v, sel_channels=selc, sel_pages=selp)
        rkv.rkv_check_status(ws)
        res[mode] = (out, selp, selc)
    return res


def _same(res, tag):
    oc, pc, cc = res["c"]
    om, pm, cm = res["m"]
    assert torch.equal(pc, pm), f"{tag}: selected pages differ"
    assert torch.equal(cc, cm), f"{tag}: selected channels differ"
    assert torch.equal(oc, om), f"{tag}: outputs differ"


def test_mt_equals_compact_path():
    # two prompts that stage 1 really filters (9000, 7000 tokens -> 4096 kept) and one short
    # enough for the dense path (200 <= budget)
    st = _setup([9000, 7000, 200], steps=0, seed=6100)
    assert torch.equal(st["kmin_c"], st["kmin_m"]) and torch.equal(st["kmax_c"], st["kmax_m"])
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    dq = S.decode_queries(st["wl"], 3, seed=6150, device="cuda")
    for t in range(3):
        _same(_step(st, dq[t]), f"step {t}")


def test_mt_appends_equal_compact_path():
    steps = 12
    st = _setup([9000, 7000, 200], steps=steps, seed=6200)
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    dq = S.decode_queries(st["wl"], steps, seed=6250, device="cuda")
    nk, nv = S.append_tokens(st["wl"], steps, st["x"]["sigma"], seed=6290, device="cuda")
    lens0 = st["x"]["seq_lens"].cpu().numpy().copy()
    kept0 = st["kept_len"].cpu().numpy().copy()
    for t in range(steps):
        _same(_step(st, dq[t], nk[t], nv[t]), f"step {t}")
    assert np.array_equal(st["full_len"].cpu().numpy(), lens0 + steps)
    assert np.array_equal(st["kept_len"].cpu().numpy(), kept0 + steps)
    assert torch.equal(st["kmin_c"], st["kmin_m"]) and torch.equal(st["kmax_c"], st["kmax_m"])
    kept = st["kept"].cpu().numpy()
    for u in range(st["wl"].n):
        L, n1 = int(lens0[u]), int(kept0[u])
        for g in range(st["wl"].n_kv):
            assert np.array_equal(kept[u, g, n1:n1 + steps], np.arange(L, L + steps))
            assert torch.equal(st["k_f"][u, g, L:L + steps], nk[:, u, g])
            assert torch.equal(st["v_f"][u, g, L:L + steps], nv[:, u, g])


def test_mt_against_oracle():
    st = _setup([9000, 7000, 200], steps=0, seed=6300)
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    dq = S.decode_queries(st["wl"], 1, seed=6350, device="cuda")
    res = _step(st, dq[0])
    out, selp, _ = res["m"]
    gqa = st["wl"].gqa
    for (u, g) in [(0, 1), (1, 0), (2, 1)]:
        L = int(st["full_len"][u])
        n1 = int(st["kept_len"][u])
        kf, vf = _f64(st["k_f"][u, g, :L]), _f64(st["v_f"][u, g, :L])
        kept = st["kept"][u, g, :n1].cpu().numpy()
        kmin, kmax = O.mt_page_summaries(kf, kept, n1, PAGE)
        qh = _f64(dq[0, u, g * gqa:(g + 1) * gqa])
        ref = O.mt_hybrid_decode(qh, kf, vf, kept, n1, kmin, kmax, BUDGET, PAGE, CHANNELS,
                                 st["scale"])
        tag = f"unit {u} kv {g}"
        if ref["pages"] is None:
            parity.check_attention(_f64(out[u, g * gqa:(g + 1) * gqa]), qh, kf[kept[:n1]],
                                   vf[kept[:n1]], st["scale"], tag)
            continue
        gp = selp[u, g].cpu().numpy()
        parity.check_selection(gp, ref["scores"], len(ref["pages"]), tag)
        rows = np.concatenate([kept[p * PAGE:min(n1, (p + 1) * PAGE)] for p in gp])
        parity.check_attention(_f64(out[u, g * gqa:(g + 1) * gqa]), qh, kf[rows], vf[rows],
                               st["scale"], tag)


def test_mt_bad_kept_index_sets_status():
    # the kernels check every kept index before using it: an out-of-range entry is reported
    # (RKV_DEV_BAD_INDEX) and row 0 is read in its place
    from sparse_kv_cache_snapkv_gb300 import rkv
    st = _setup([9000, 7000, 200], steps=0, seed=6400)
    kept = st["kept"]
    kept[0, 0, 5] = st["k_f"].shape[2] + 100
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_check_status(rkv.rkv_build_page_summaries_mt(st["k_f"], kept, st["kept_len"],
                                                             PAGE, st["kmin_m"], st["kmax_m"]))
    assert e.value.bits & 0x10
    # the decode reads it only if its page is selected: make that certain with the dense path
    # over a kept list of 200 tokens that includes the bad entry
    kept[2, 0, 7] = -3
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    dq = S.decode_queries(st["wl"], 1, seed=6450, device="cuda")
    out = torch.empty_like(dq[0])
    ws = rkv.rkv_hybrid_decode_mt(dq[0], st["k_f"], st["v_f"], st["full_len"], kept,
                                  st["kept_len"], st["kmin_m"], st["kmax_m"], BUDGET, PAGE,
                                  CHANNELS, st["scale"], out)
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_check_status(ws)
    assert e.value.bits & 0x10
    assert torch.isfinite(out.float()).all()


def test_mt_second_turn_refilter():
    # two turns of RocketKV-MT: turn 1 filters the prompt (index only: nothing is evicted),
    # decodes with appends; turn 2 appends its new input to the full cache, filters the whole
    # history again with its own window queries, rebuilds the summaries and decodes on
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    rkv.load()
    T1, T2, M = 8, 4, 256
    wl = S.Workload("mt2", 2, 1, 2, 4, D, (9000, 7000), W, BUDGET, needles=8)
    x = S.prefill_inputs(wl, seed=6500, device="cuda")
    t2 = S.second_turn_inputs(wl, x, M, 8, seed=6510, device="cuda")
    nk, nv = S.append_tokens(wl, T1 + T2, x["sigma"], seed=6520, device="cuda")
    dq = S.decode_queries(wl, T1 + T2, seed=6530, device="cuda")
    n, n_kv, gqa, max_len = wl.n, wl.n_kv, wl.gqa, wl.max_len
    keep = rkv.rkv_plan(max_len, BUDGET)[0]
    kcap = keep + T1 + T2
    full_cap = max_len + T1 + M + T2
    page_cap = ((kcap + PAGE - 1) // PAGE + 7) // 8 * 8
    scale = 1.0 / math.sqrt(D)
    k_f = torch.zeros(n, n_kv, full_cap, D, dtype=torch.bfloat16, device="cuda")
    v_f = torch.zeros_like(k_f)
    k_f[:, :, :max_len] = x["k"]
    v_f[:, :, :max_len] = x["v"]
    full_len = x["seq_lens"].clone()
    kept = torch.full((n, n_kv, kcap), -7, dtype=torch.int32, device="cuda")
    kept_len = torch.empty(n, dtype=torch.int32, device="cuda")
    kmin = torch.zeros(n, n_kv, D, page_cap, dtype=torch.bfloat16, device="cuda")
    kmax = torch.zeros_like(kmin)

    def decode(t):
        out = torch.empty_like(dq[t])
        selp = torch.empty(n, n_kv, (BUDGET // 2) // PAGE, dtype=torch.int32, device="cuda")
        ws = rkv.rkv_hybrid_decode_mt(dq[t], k_f, v_f, full_len, kept, kept_len, kmin, kmax,
                                      BUDGET, PAGE, CHANNELS, scale, out, new_k=nk[t],
                                      new_v=nv[t], sel_pages=selp)
        rkv.rkv_check_status(ws)
        return out, selp

    # ---- turn 1
    rkv.rkv_check_status(rkv.rkv_snapkv_select(k_f, full_len, x["q_win"], 0, keep, scale, kept,
                                               kept_len))
    assert (kept[:, :, keep:] == -7).all(), "entries past keep must stay untouched"
    kept1 = kept[:, :, :keep].cpu().numpy().copy()
    rkv.rkv_check_status(rkv.rkv_build_page_summaries_mt(k_f, kept, kept_len, PAGE, kmin, kmax))
    for t in range(T1):
        decode(t)
    # ---- turn 2: the new input goes to the end of the full cache, then the history is filtered
    for u in range(n):
        L = int(full_len[u])
        k_f[u, :, L:L + M] = t2["new_k"][u]
        v_f[u, :, L:L + M] = t2["new_v"][u]
    full_len += M
    rkv.rkv_check_status(rkv.rkv_snapkv_select(k_f, full_len, t2["q_win"], 0, keep, scale, kept,
                                               kept_len))
    kept2 = kept[:, :, :keep].cpu().numpy().copy()
    assert np.array_equal(kept_len.cpu().numpy(), [keep, keep])
    kmin.zero_()
    kmax.zero_()
    rkv.rkv_check_status(rkv.rkv_build_page_summaries_mt(k_f, kept, kept_len, PAGE, kmin, kmax))
    hist_len = full_len.cpu().numpy().copy()
    for u in range(n):
        for g in range(n_kv):
            tag = f"unit {u} kv {g}"
            L2 = int(hist_len[u])
            hist = _f64(k_f[u, g, :L2])
            q2 = _f64(t2["q_win"][u, g * gqa:(g + 1) * gqa])
            kk = O.adaptive_kernel_size(L2)
            pooled = O.pool_max(O.window_scores(hist, q2, scale), kk)
            assert np.array_equal(kept2[u, g, keep - W:], np.arange(L2 - W, L2)), tag
            parity.check_selection(kept2[u, g, :keep - W], pooled, keep - W, tag)
            n2 = t2["needles"][u, g].numpy()
            assert np.isin(n2, kept2[u, g]).all(), f"{tag}: turn 2 misses its keys"
            assert not np.isin(n2, kept1[u, g]).all(), f"{tag}: turn 1 kept every turn-2 key"
    # ---- turn 2 decodes on the new kept list (with appends) and matches the oracle
    for t in range(T1, T1 + T2 - 1):
        decode(t)
    t = T1 + T2 - 1
    kept_before = kept_len.cpu().numpy().copy()
    len_before = full_len.cpu().numpy().copy()
    out, selp = decode(t)
    for u in range(n):
        for g in range(n_kv):
            tag = f"turn 2 decode unit {u} kv {g}"
            L, n1 = int(len_before[u]), int(kept_before[u])
            kf = _f64(k_f[u, g, :L + 1])
            vf = _f64(v_f[u, g, :L + 1])
            kl = kept[u, g, :n1 + 1].cpu().numpy()
            assert kl[n1] == L, tag
            assert np.array_equal(kl[keep:n1], np.arange(len_before[u] - (n1 - keep), L)), tag
            mn, mx = O.mt_page_summaries(kf, kl, n1 + 1, PAGE)
            qh = _f64(dq[t, u, g * gqa:(g + 1) * gqa])
            ref = O.mt_hybrid_decode(qh, kf, vf, kl, n1 + 1, mn, mx, BUDGET, PAGE, CHANNELS,
                                     scale)
            gp = selp[u, g].cpu().numpy()
            parity.check_selection(gp, ref["scores"], len(ref["pages"]), tag)
            rows = np.concatenate([kl[p * PAGE:min(n1 + 1, (p + 1) * PAGE)] for p in gp])
            parity.check_attention(_f64(out[u, g * gqa:(g + 1) * gqa]), qh, kf[rows], vf[rows],
                                   scale, tag)
