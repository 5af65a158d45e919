"""Parity of SnapKV++ compression (tensor-core window scores, pooling + top-k, gather) against the
CPU oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

from oracle import rocketkv as O
from tests import parity

pytestmark = pytest.mark.gpu

D = 128
SCORE_REL = 1e-4


def _lib():
    from sparse_kv_cache_snapkv_gb300 import rkv
    rkv.load()
    return rkv


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _inputs(n_seq, n_kv, gqa, lens, window, seed, needles=0, outliers=0, layers=1):
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    wl = S.Workload("t", n_seq, layers, n_kv, gqa, D, tuple(lens), window, 256,
                    needles=needles, outliers=outliers)
    x = S.prefill_inputs(wl, seed=seed, device="cuda")
    return wl, x


def _run(rkv, x, window, kernel, keep, cap=None, avg=False):
    k, v, q, lens = x["k"], x["v"], x["q_win"], x["seq_lens"]
    n, n_kv, max_len, _ = k.shape
    cap = cap or keep
    k_out = torch.zeros(n, n_kv, cap, D, dtype=torch.bfloat16, device="cuda")
    v_out = torch.zeros_like(k_out)
    kept = torch.full((n, n_kv, keep), -9, dtype=torch.int32, device="cuda")
    out_len = torch.full((n,), -9, dtype=torch.int32, device="cuda")
    scores = torch.full((n, n_kv, max_len - window), -1.0, dtype=torch.float32, device="cuda")
    fn = rkv.rkv_snapkv_compress_avg_pool if avg else rkv.rkv_snapkv_compress
    ws = fn(k, v, lens, q, kernel, keep, 1.0 / math.sqrt(D), k_out, v_out, kept, out_len,
            scores_out=scores)
    rkv.rkv_check_status(ws)
    return k_out, v_out, kept, out_len, scores


def _check_unit(x, u, g, gqa, window, kernel, keep, k_out, v_out, kept, out_len, scores,
                tag="", pool=O.pool_max):
    L = int(x["seq_lens"][u])
    W = window
    k = _f64(x["k"][u, g, :L])
    v = _f64(x["v"][u, g, :L])
    q = _f64(x["q_win"][u, g * gqa:(g + 1) * gqa])
    ref_scores = O.window_scores(k, q, 1.0 / math.sqrt(D))
    gs = scores[u, g, :L - W].cpu().numpy().astype(np.float64)
    err = np.abs(gs - ref_scores)
    tol = SCORE_REL * np.abs(ref_scores) + 1e-30
    assert (err <= tol).all(), (f"{tag} scores: {(err > tol).sum()} bad, worst rel "
                                f"{(err / np.maximum(ref_scores, 1e-30)).max():.2e}")
    kk = kernel if kernel > 0 else O.adaptive_kernel_size(L)
    pooled = pool(ref_scores, kk)
    got = kept[u, g].cpu().numpy()
    cnt = min(L, keep)
    assert int(out_len[u]) == cnt, tag
    assert (got[cnt:] == -1).all(), tag
    if L <= keep:
        assert np.array_equal(got[:L], np.arange(L)), tag
    else:
        assert np.array_equal(got[keep - W:keep], np.arange(L - W, L)), f"{tag} window"
        pre = got[:keep - W]
        assert np.all(np.diff(pre) > 0), f"{tag} not ascending"
        parity.check_selection(pre, pooled, keep - W, f"{tag} kept")
    idx = got[:cnt]
    assert np.array_equal(_f64(k_out[u, g, :cnt]), k[idx]), f"{tag} gathered K"
    assert np.array_equal(_f64(v_out[u, g, :cnt]), v[idx]), f"{tag} gathered V"


@pytest.mark.parametrize("keep", [256, 1024, 4096])
def test_snapkv_tiny_config(keep):
    # batch 1, 8 q / 2 kv heads, 4K prompt, W 32, pooling 7, 8 planted needles
    rkv = _lib()
    wl, x = _inputs(1, 2, 4, [4096], 32, seed=101, needles=8)
    res = _run(rkv, x, 32, 7, keep)
    for g in range(2):
        _check_unit(x, 0, g, 4, 32, 7, keep, *res, tag=f"keep {keep} kv {g}")
    if keep == 256:
        kept = res[2].cpu().numpy()
        for g in range(2):
            assert set(x["needles"][0, g].tolist()) <= set(kept[0, g].tolist())


def test_snapkv_window64_rows256_ragged():
    # G * W = 256 (two 128-row blocks), ragged lengths incl. one <= keep and one not tile-aligned
    rkv = _lib()
    wl, x = _inputs(3, 2, 4, [5000, 700, 3333], 64, seed=102, needles=4)
    res = _run(rkv, x, 64, 15, 1024)
    for u in range(3):
        for g in range(2):
            _check_unit(x, u, g, 4, 64, 15, 1024, *res, tag=f"u{u} g{g}")


@pytest.mark.parametrize("gqa,window", [(1, 32), (2, 48), (8, 16), (4, 5)])
def test_snapkv_row_padding(gqa, window):
    # G * W below 128 / between 128 and 256: padded query rows must not leak into the scores
    rkv = _lib()
    wl, x = _inputs(2, 2, gqa, [2047, 1500], window, seed=103 + gqa)
    res = _run(rkv, x, window, 3, 512)
    for u in range(2):
        for g in range(2):
            _check_unit(x, u, g, gqa, window, 3, 512, *res, tag=f"gqa{gqa} u{u} g{g}")


def test_snapkv_adaptive_kernel_and_long_prompt():
    # one 40K prompt (kernel 31 by the length rule) and one 9K prompt (kernel 15), many splits
    rkv = _lib()
    wl, x = _inputs(2, 1, 4, [40000, 9000], 32, seed=104, needles=16)
    res = _run(rkv, x, 32, 0, 2048)
    for u in range(2):
        _check_unit(x, u, 0, 4, 32, 0, 2048, *res, tag=f"u{u}")


@pytest.mark.parametrize("kernel", [1, 5, 31, 0])
def test_snapkv_select_paths(kernel):
    # the whole-unit shared-memory select (at most 32768 scores, pooling kernel 2^k - 1) at its
    # size limit (32800 - 32 = 32768 scores), on ragged lengths and with a kernel wider than the
    # 32 positions a thread owns; kernel 5 takes the general select
    rkv = _lib()
    wl, x = _inputs(3, 1, 4, [32800, 12345, 9000], 32, seed=107, needles=8)
    res = _run(rkv, x, 32, kernel, 2048)
    for u in range(3):
        _check_unit(x, u, 0, 4, 32, kernel, 2048, *res, tag=f"kernel {kernel} u{u}")


def _fixed_point_avg(scores, kernel):
    """The select's average pooling restated on its own fp32 scores: 32.32 fixed-point window
    sums (exact), then float(sum) * 2^-32 / count in fp32."""
    fx = np.rint(scores.astype(np.float64) * 2.0 ** 32).astype(np.int64)
    c = np.concatenate([[0], np.cumsum(fx)])
    n, r = fx.shape[0], kernel // 2
    i = np.arange(n)
    lo, hi = np.maximum(0, i - r), np.minimum(n - 1, i + r)
    s = (c[hi + 1] - c[lo]).astype(np.float32) * np.float32(2.0 ** -32)
    return s / (hi - lo + 1).astype(np.float32)


@pytest.mark.parametrize("lens,kernel", [((32800, 12345, 9000), 7), ((32800, 12345, 9000), 15),
                                         ((32800, 12345, 9000), 5), ((32800, 12345, 9000), 0),
                                         ((40000, 5000, 2100), 5), ((40000, 5000, 2100), 0)])
def test_snapkv_avg_pool(lens, kernel):
    # average pooling over the clipped window: the shared-memory select (every odd kernel when
    # all units hold at most 32768 scores) and the general select (a 40000-token prompt); ragged
    # lengths, one prompt barely above keep
    rkv = _lib()
    W, keep = 32, 2048
    wl, x = _inputs(3, 1, 4, list(lens), W, seed=109, needles=8)
    res = _run(rkv, x, W, kernel, keep, avg=True)
    kept, scores = res[2].cpu().numpy(), res[4].cpu().numpy()
    for u in range(3):
        _check_unit(x, u, 0, 4, W, kernel, keep, *res, tag=f"avg kernel {kernel} u{u}",
                    pool=O.pool_avg)
        # exact: the kept set is the top-k (ties -> lower position) of the fixed-point means
        # of the kernel's own scores
        L = lens[u]
        kk = kernel if kernel > 0 else O.adaptive_kernel_size(L)
        keys = _fixed_point_avg(scores[u, 0, :L - W], kk).astype(np.float64)
        order = np.lexsort((np.arange(L - W), -keys))
        assert np.array_equal(kept[u, 0, :keep - W], np.sort(order[:keep - W])), f"u{u} exact"
    # average and max pooling keep different sets
    res_max = _run(rkv, x, W, kernel, keep)
    assert not torch.equal(res[2], res_max[2])


@pytest.mark.parametrize("kernel", [1, 3, 7, 15, 31])
def test_snapkv_select_tiny_prefixes(kernel):
    # prefixes of 8, 33 and 68 scores: one, two and three threads of the shared-memory select
    # hold positions, so the register pooling's neighbour exchange meets the end of the scores
    # inside a warp; pooling windows wider than the prefix clip at both ends
    rkv = _lib()
    W, keep = 32, 36
    wl, x = _inputs(3, 1, 4, [40, 65, 100], W, seed=110, needles=0)
    res = _run(rkv, x, W, kernel, keep)
    for u in range(3):
        _check_unit(x, u, 0, 4, W, kernel, keep, *res, tag=f"kernel {kernel} u{u}")


def test_snapkv_per_head_without_group_sum():
    # SnapKV without the GQA enhancement: each query head is scored with its own window rows and
    # keeps its own rows of its K/V head; ragged lengths, one prompt shorter than keep
    rkv = _lib()
    gqa, W, keep, kernel = 4, 32, 1024, 15
    wl, x = _inputs(3, 2, gqa, [5000, 3001, 900], W, seed=108, needles=4)
    k, v, q, lens = x["k"], x["v"], x["q_win"], x["seq_lens"]
    n, n_kv, max_len, _ = k.shape
    hq = n_kv * gqa
    scale = 1.0 / math.sqrt(D)
    k_out = torch.zeros(n, hq, keep, D, dtype=torch.bfloat16, device="cuda")
    v_out = torch.zeros_like(k_out)
    kept = torch.full((n, hq, keep), -9, dtype=torch.int32, device="cuda")
    out_len = torch.full((n,), -9, dtype=torch.int32, device="cuda")
    scores = torch.full((n, hq, max_len - W), -1.0, dtype=torch.float32, device="cuda")
    ws = rkv.rkv_snapkv_compress_per_head(k, v, lens, q, kernel, keep, scale, k_out, v_out, kept,
                                          out_len, scores_out=scores)
    rkv.rkv_check_status(ws)
    for (u, h) in [(0, 0), (0, 5), (1, 3), (1, 6), (2, 2)]:
        g, L = h // gqa, int(lens[u])
        tag = f"unit {u} q head {h}"
        kk, vv = _f64(k[u, g, :L]), _f64(v[u, g, :L])
        ref = O.window_scores(kk, _f64(q[u, h:h + 1]), scale)
        gs = scores[u, h, :L - W].cpu().numpy().astype(np.float64)
        assert (np.abs(gs - ref) <= SCORE_REL * np.abs(ref) + 1e-30).all(), tag
        got = kept[u, h].cpu().numpy()
        cnt = min(L, keep)
        assert int(out_len[u]) == cnt, tag
        if L <= keep:
            assert np.array_equal(got[:L], np.arange(L)), tag
        else:
            assert np.array_equal(got[keep - W:], np.arange(L - W, L)), tag
            parity.check_selection(got[:keep - W], O.pool_max(ref, kernel), keep - W, tag)
        idx = got[:cnt]
        assert np.array_equal(_f64(k_out[u, h, :cnt]), kk[idx]), tag
        assert np.array_equal(_f64(v_out[u, h, :cnt]), vv[idx]), tag
    # heads of one group select differently (they are no longer summed)
    assert not torch.equal(kept[0, 0], kept[0, 1])


@pytest.mark.parametrize("page", [1, 4, 16, 64])
def test_snapkv_summarized_equals_separate_summaries(page):
    # the gather's page summaries equal compress + rkv_build_page_summaries bit for bit: ragged
    # lengths (partial last pages), one prompt shorter than keep, one shorter than the window
    rkv = _lib()
    wl, x = _inputs(4, 2, 4, [5000, 3001, 1030, 20], 32, seed=109)
    k, v, q, lens = x["k"], x["v"], x["q_win"], x["seq_lens"]
    n, n_kv, max_len, _ = k.shape
    keep = 1024
    page_cap = ((keep + page - 1) // page + 7) // 8 * 8
    scale = 1.0 / math.sqrt(D)
    outs = []
    for fused in (False, True):
        k_out = torch.zeros(n, n_kv, keep, D, dtype=torch.bfloat16, device="cuda")
        v_out = torch.zeros_like(k_out)
        kept = torch.empty(n, n_kv, keep, dtype=torch.int32, device="cuda")
        out_len = torch.empty(n, dtype=torch.int32, device="cuda")
        kmin = torch.full((n, n_kv, D, page_cap), 7.0, dtype=torch.bfloat16, device="cuda")
        kmax = torch.full_like(kmin, 7.0)
        def status(ws):
            try:
                rkv.rkv_check_status(ws)
            except rkv.RkvError as e:
                assert e.bits == 0x2, e  # only the prompt shorter than the window is flagged

        if fused:
            status(rkv.rkv_snapkv_compress_summarized(k, v, lens, q, 7, keep, scale, k_out,
                                                      v_out, kept, out_len, page, kmin, kmax))
        else:
            status(rkv.rkv_snapkv_compress(k, v, lens, q, 7, keep, scale, k_out, v_out, kept,
                                           out_len))
            status(rkv.rkv_build_page_summaries(k_out, out_len, page, kmin, kmax))
        outs.append((k_out, kept, out_len, kmin, kmax))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_snapkv_multiple_waves():
    # 6 units of 64K tokens: K of all units exceeds one L2-sized wave, so several waves run
    rkv = _lib()
    wl, x = _inputs(6, 1, 4, [65536, 65536, 60001, 65536, 1000, 65536], 32, seed=105)
    res = _run(rkv, x, 32, 31, 4096)
    for u in (0, 2, 4, 5):
        _check_unit(x, u, 0, 4, 32, 31, 4096, *res, tag=f"u{u}")


def test_snapkv_outlier_channels_128k_sample():
    # 128K prompt with 4 outlier channels at 10x (large logits), budget 1024 -> keep 16384
    rkv = _lib()
    wl, x = _inputs(1, 2, 4, [131072], 32, seed=106, needles=64, outliers=4)
    res = _run(rkv, x, 32, 31, 16384)
    for g in range(2):
        _check_unit(x, 0, g, 4, 32, 31, 16384, *res, tag=f"g{g}")


def test_snapkv_scores_only_matches_oracle():
    # the score passes alone: ragged lengths (one not tile-aligned), G * W = 128 and 256; the
    # entries past a unit's L - W stay untouched
    rkv = _lib()
    for window, lens in ((32, [3001, 700]), (64, [5000, 1999])):
        wl, x = _inputs(2, 2, 4, lens, window, seed=150 + window, needles=2)
        n, n_kv, max_len, _ = x["k"].shape
        scores = torch.full((n, n_kv, max_len - window), -3.0, dtype=torch.float32,
                            device="cuda")
        ws = rkv.rkv_snapkv_scores(x["k"], x["seq_lens"], x["q_win"], 1.0 / math.sqrt(D), scores)
        rkv.rkv_check_status(ws)
        for u, L in enumerate(lens):
            for g in range(n_kv):
                k = _f64(x["k"][u, g, :L])
                q = _f64(x["q_win"][u, g * 4:(g + 1) * 4])
                ref = O.window_scores(k, q, 1.0 / math.sqrt(D))
                gs = scores[u, g, :L - window].cpu().numpy().astype(np.float64)
                err = np.abs(gs - ref)
                assert (err <= SCORE_REL * np.abs(ref) + 1e-30).all(), f"W {window} unit {u}"
                assert (scores[u, g, L - window:] == -3.0).all(), f"W {window} unit {u} tail"
