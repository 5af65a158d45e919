"""Paged (block-table) compact cache through the C ABI.

Stage 1 writes its kept rows straight into blocks of a shared pool; the summaries and the decode
(appends included) read and write them through the table. The pages describe no paging: it is a
storage layout, so every result must equal the contiguous calls' bit for bit, and (a separate
test) what the oracle computes from the inputs when the pool is read back through the oracle's
own view of the block table. The table is a
random permutation of pool blocks and every block or row the table does not name holds NaN, so a
read from a wrong block shows up in the outputs. Block sizes 2 (a 4-token page spans two blocks)
and 64.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

D = 128
W = 32
BUDGET = 256
PAGE = 4
CHANNELS = 32


def _gather_pool(pool, table, u, g, n_tok):
    block = pool.shape[2]
    t = torch.arange(n_tok, device=pool.device)
    return pool[table[u].long()[t // block], g, t % block]


def _setup(block, steps, seed):
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    rkv.load()
    wl = S.Workload("paged", 3, 1, 2, 4, D, (9000, 5000, 200), W, BUDGET, needles=8)
    x = S.prefill_inputs(wl, seed=seed, device="cuda")
    n, n_kv, max_len = wl.n, wl.n_kv, wl.max_len
    keep = rkv.rkv_plan(max_len, BUDGET)[0]
    cap = keep + steps
    max_blocks = (cap + block - 1) // block
    num_blocks = n * max_blocks + 17
    page_cap = ((cap + PAGE - 1) // PAGE + 7) // 8 * 8
    scale = 1.0 / math.sqrt(D)
    gen = torch.Generator().manual_seed(seed + 1)
    perm = torch.randperm(num_blocks, generator=gen)[: n * max_blocks]
    table = perm.view(n, max_blocks).to(torch.int32).cuda()
    st = {"rkv": rkv, "x": x, "wl": wl, "keep": keep, "cap": cap, "scale": scale, "table": table,
          "page_cap": page_cap}
    # contiguous compact cache
    st["k_c"] = torch.zeros(n, n_kv, cap, D, dtype=torch.bfloat16, device="cuda")
    st["v_c"] = torch.zeros_like(st["k_c"])
    kept_c = torch.empty(n, n_kv, keep, dtype=torch.int32, device="cuda")
    st["len_c"] = torch.empty(n, dtype=torch.int32, device="cuda")
    rkv.rkv_check_status(rkv.rkv_snapkv_compress(x["k"], x["v"], x["seq_lens"], x["q_win"], 0,
                                                 keep, scale, st["k_c"], st["v_c"], kept_c,
                                                 st["len_c"]))
    # paged: pools full of NaN, then stage 1 through the table
    st["k_p"] = torch.full((num_blocks, n_kv, block, D), float("nan"), dtype=torch.bfloat16,
                           device="cuda")
    st["v_p"] = torch.full_like(st["k_p"], float("nan"))
    kept_p = torch.empty_like(kept_c)
    st["len_p"] = torch.empty_like(st["len_c"])
    rkv.rkv_check_status(rkv.rkv_snapkv_compress_paged(x["k"], x["v"], x["seq_lens"], x["q_win"],
                                                       0, keep, scale, st["k_p"], st["v_p"], table,
                                                       kept_p, st["len_p"]))
    assert torch.equal(kept_c, kept_p) and torch.equal(st["len_c"], st["len_p"])
    st["kept_p"] = kept_p
    z = lambda: torch.zeros(n, n_kv, D, page_cap, dtype=torch.bfloat16, device="cuda")
    st["kmin_c"], st["kmax_c"], st["kmin_p"], st["kmax_p"] = z(), z(), z(), z()
    rkv.rkv_check_status(rkv.rkv_build_page_summaries(st["k_c"], st["len_c"], PAGE, st["kmin_c"],
                                                      st["kmax_c"]))
    rkv.rkv_check_status(rkv.rkv_build_page_summaries_paged(st["k_p"], table, st["len_p"], PAGE,
                                                            st["kmin_p"], st["kmax_p"]))
    return st


def _check_rows(st):
    wl = st["wl"]
    for u in range(wl.n):
        L = int(st["len_c"][u])
        for g in range(wl.n_kv):
            assert torch.equal(_gather_pool(st["k_p"], st["table"], u, g, L), st["k_c"][u, g, :L])
            assert torch.equal(_gather_pool(st["v_p"], st["table"], u, g, L), st["v_c"][u, g, :L])
    assert torch.equal(st["kmin_c"], st["kmin_p"]) and torch.equal(st["kmax_c"], st["kmax_p"])


def _step(st, q, new_k=None, new_v=None):
    rkv = st["rkv"]
    n, n_kv = st["wl"].n, st["wl"].n_kv
    res = []
    for paged in (False, True):
        out = torch.empty_like(q)
        selp = torch.empty(n, n_kv, (BUDGET // 2) // PAGE, dtype=torch.int32, device="cuda")
        if paged:
            ws = rkv.rkv_hybrid_decode_paged(q, st["k_p"], st["v_p"], st["table"], st["len_p"],
                                             st["kmin_p"], st["kmax_p"], BUDGET, PAGE, CHANNELS,
                                             st["scale"], out, new_k=new_k, new_v=new_v,
                                             sel_pages=selp)
        else:
            ws = rkv.rkv_hybrid_decode(q, st["k_c"], st["v_c"], st["len_c"], st["kmin_c"],
                                       st["kmax_c"], BUDGET, PAGE, CHANNELS, st["scale"], out,
                                       new_k=new_k, new_v=new_v, sel_pages=selp)
        rkv.rkv_check_status(ws)
        res.append((out, selp))
    assert torch.equal(res[0][1], res[1][1]), "selected pages differ"
    assert torch.isfinite(res[1][0].float()).all(), "a NaN row was read"
    assert torch.equal(res[0][0], res[1][0]), "outputs differ"


@pytest.mark.parametrize("block", [2, 64])
def test_paged_equals_contiguous(block):
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    steps = 10
    st = _setup(block, steps, seed=7100 + block)
    _check_rows(st)
    dq = S.decode_queries(st["wl"], 3 + steps, seed=7150, device="cuda")
    for t in range(3):
        _step(st, dq[t])
    nk, nv = S.append_tokens(st["wl"], steps, st["x"]["sigma"], seed=7190, device="cuda")
    for t in range(steps):
        _step(st, dq[3 + t], nk[t], nv[t])
    assert torch.equal(st["len_c"], st["len_p"])
    _check_rows(st)


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("block", [2, 64])
def test_paged_against_oracle(block):
    """The paged path against the oracle, not against the contiguous GPU path.

    Every row the paged pool holds is read back through the oracle's own view of a block table
    (O.paged_view) and must equal the row the oracle derives from the inputs: the prompt row of
    each kept index (the kept set itself checked against O.snapkv_compress within the tie band),
    then every appended token. The page summaries must equal O.page_summaries of those rows bit
    for bit, and each decode step's channels, approximate scores, pages and outputs must match
    O.hybrid_decode with the acceptance rules of the other parity tests, with and without
    appends.
    """
    from oracle import rocketkv as O
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    from tests import parity
    steps = 5
    st = _setup(block, steps, seed=7400 + block)
    rkv, wl, x, keep, scale = st["rkv"], st["wl"], st["x"], st["keep"], st["scale"]
    n, n_kv, G = wl.n, wl.n_kv, wl.gqa
    table = st["table"].cpu().numpy()
    kept = st["kept_p"].cpu().numpy()
    S_pages = (BUDGET // 2) // PAGE
    # oracle rows per (unit, KV head), from the inputs only
    rows = {}
    for u in range(n):
        L = int(x["seq_lens"][u])
        for g in range(n_kv):
            k = _f64(x["k"][u, g, :L])
            v = _f64(x["v"][u, g, :L])
            tag = f"block {block} unit {u} kv {g}"
            cnt = min(L, keep)
            got = kept[u, g, :cnt]
            if L > keep:
                q = _f64(x["q_win"][u, g * G:(g + 1) * G])
                pooled = O.snapkv_compress(k, v, q, keep, O.adaptive_kernel_size(L), scale)[4]
                assert np.array_equal(got[keep - W:], np.arange(L - W, L)), f"{tag} window"
                parity.check_selection(got[:keep - W], pooled, keep - W, f"{tag} kept")
            else:
                assert np.array_equal(got, np.arange(L)), tag
            rows[(u, g)] = (k[got], v[got])

    def check_state(step):
        kp, vp = _f64(st["k_p"]), _f64(st["v_p"])
        kmin, kmax = _f64(st["kmin_p"]), _f64(st["kmax_p"])
        lens = st["len_p"].cpu().numpy()
        for (u, g), (kc, vc) in rows.items():
            tag = f"block {block} step {step} unit {u} kv {g}"
            L = int(lens[u])
            assert L == kc.shape[0], tag
            assert np.array_equal(O.paged_view(kp, table[u], L, g), kc), f"{tag} K rows"
            assert np.array_equal(O.paged_view(vp, table[u], L, g), vc), f"{tag} V rows"
            rmin, rmax = O.page_summaries(kc, L, PAGE)
            P = rmin.shape[1]
            assert np.array_equal(kmin[u, g, :, :P], rmin), f"{tag} Kmin"
            assert np.array_equal(kmax[u, g, :, :P], rmax), f"{tag} Kmax"

    check_state("prefill")
    dq = S.decode_queries(wl, 2 + steps, seed=7450, device="cuda")
    nk, nv = S.append_tokens(wl, steps, x["sigma"], seed=7490, device="cuda")
    for t in range(2 + steps):
        app = t >= 2
        q = dq[t]
        if app:
            a_k, a_v = nk[t - 2], nv[t - 2]
            for (u, g), (kc, vc) in list(rows.items()):
                rows[(u, g)] = (np.concatenate([kc, _f64(a_k[u, g])[None]]),
                                np.concatenate([vc, _f64(a_v[u, g])[None]]))
        out = torch.empty_like(q)
        sel_c = torch.full((n, n_kv, CHANNELS), -7, dtype=torch.int32, device="cuda")
        sel_p = torch.full((n, n_kv, S_pages), -7, dtype=torch.int32, device="cuda")
        approx = torch.zeros(n, n_kv, st["page_cap"], dtype=torch.float32, device="cuda")
        ws = rkv.rkv_hybrid_decode_paged(q, st["k_p"], st["v_p"], st["table"], st["len_p"],
                                         st["kmin_p"], st["kmax_p"], BUDGET, PAGE, CHANNELS,
                                         scale, out, new_k=a_k if app else None,
                                         new_v=a_v if app else None, sel_channels=sel_c,
                                         sel_pages=sel_p, approx_scores=approx)
        rkv.rkv_check_status(ws)
        check_state(t)
        qq = _f64(q)
        for (u, g), (kc, vc) in rows.items():
            tag = f"block {block} step {t} unit {u} kv {g}"
            L = kc.shape[0]
            qh = qq[u, g * G:(g + 1) * G]
            rmin, rmax = O.page_summaries(kc, L, PAGE)
            ref = O.hybrid_decode(qh, kc, vc, L, rmin, rmax, BUDGET, PAGE, CHANNELS, scale)
            gout = _f64(out[u, g * G:(g + 1) * G])
            if ref["channels"] is None:
                assert (sel_p[u, g] == -1).all(), tag
                parity.check_attention(gout, qh, kc[:L], vc[:L], scale, tag)
                continue
            parity.check_selection(sel_c[u, g].cpu().numpy(), np.abs(qh).sum(axis=0), CHANNELS,
                                   f"{tag} channels")
            gch = np.sort(sel_c[u, g].cpu().numpy())
            q_g = qh.sum(axis=0)
            ref_a = O.approx_scores(q_g, gch, rmin, rmax)
            P = rmin.shape[1]
            parity.check_approx(approx[u, g, :P].cpu().numpy(), ref_a,
                                parity.approx_magnitude(q_g, gch, rmin, rmax), len(gch),
                                f"{tag} approx")
            gp = sel_p[u, g].cpu().numpy()
            nsel = min(S_pages, P)
            parity.check_selection(gp[:nsel], ref_a, nsel, f"{tag} pages")
            toks = np.concatenate([np.arange(pg * PAGE, min(L, (pg + 1) * PAGE))
                                   for pg in gp[:nsel]])
            parity.check_attention(gout, qh, kc[toks], vc[toks], scale, tag)


def test_paged_bad_table_entry_sets_status():
    from sparse_kv_cache_snapkv_gb300 import rkv
    st = _setup(64, 0, seed=7300)
    table = st["table"].clone()
    table[2, 1] = st["k_p"].shape[0] + 5      # unit 2 holds 200 tokens: block 1 is in use
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_check_status(rkv.rkv_build_page_summaries_paged(st["k_p"], table, st["len_p"],
                                                                PAGE, st["kmin_p"], st["kmax_p"]))
    assert e.value.bits & 0x10
