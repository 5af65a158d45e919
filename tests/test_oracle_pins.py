"""Pins for the CPU oracle: each check ties it to something other than itself.

The pins are the pages' worked numbers (tests/golden/*.json), closed forms, invariants, special
cases that reduce to a library routine, and brute force on tiny inputs. They run without a GPU.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.ndimage
import scipy.special
import torch

from oracle import rocketkv as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_values(shape, rng, scale=1.0):
    """Random values that are exactly representable in bf16, as float64."""
    x = torch.from_numpy(rng.standard_normal(shape) * scale).to(torch.bfloat16)
    return x.to(torch.float64).numpy()


# ---------------------------------------------------------------- planner and budget split
def test_planner_worked_example():
    g = _golden("planner_worked_example.json")
    assert g["ctx"] // g["budget"] == g["overall_ratio"]
    assert g["per_stage_ratio"] ** 2 == g["overall_ratio"]
    assert g["page"] * g["head_dim_ratio"] == g["per_stage_ratio"]
    keep, page, channels, _ = O.plan(g["ctx"], g["budget"], g["head_dim"])
    assert page == g["page"]
    assert g["head_dim"] // channels == g["head_dim_ratio"]
    assert g["ctx"] // keep == g["per_stage_ratio"]
    assert keep == g["derived_by_reading_R1"]["keep"]


def test_ratio_split_4x4():
    g = _golden("ratio_split.json")
    _, page, channels, _ = O.plan(1 << 20, 256, 128)
    assert page == g["sequence_ratio"]
    assert 128 // channels == g["head_dim_ratio"]
    assert page * (128 // channels) == g["stage2_ratio"]


@pytest.mark.parametrize("budget", [256, 512, 1024, 4096])
def test_budget_half_half(budget):
    g = _golden("budget_split.json")
    if budget == g["budget"]:
        assert budget // 2 == g["approximation_tokens"] == g["sparse_attention_tokens"]
    keep, page, channels, _ = O.plan(1 << 22, budget, 128)
    d = 128
    pages = keep // page
    approx_bytes = pages * channels * 2          # one bf16 of Kmin or Kmax per kept channel
    sparse_bytes = (budget // 2) * d * 2 * 2     # K and V rows of the B/2 exact tokens
    assert approx_bytes == sparse_bytes
    assert ((budget // 2) // page) * page == budget // 2


def test_kernel_size_monotone():
    sizes = [O.adaptive_kernel_size(L) for L in (1024, 4096, 8192, 8193, 32768, 32769, 131072)]
    assert sizes == sorted(sizes)
    assert all(s % 2 == 1 for s in sizes)
    assert O.plan(4096, 256, 128)[3] == 7


# ---------------------------------------------------------------- stage-1 scores
def _brute_scores(k, q_win, scale):
    L, d = k.shape
    G, W, _ = q_win.shape
    out = [0.0] * (L - W)
    for h in range(G):
        for j in range(W):
            vis = L - W + j + 1
            logit = [sum(q_win[h, j, c] * k[i, c] for c in range(d)) * scale for i in range(vis)]
            for i in range(L - W):
                # p_i = 1 / sum_i' exp(s_i' - s_i): no max subtraction, no vectorisation
                out[i] += 1.0 / sum(math.exp(logit[t] - logit[i]) for t in range(vis))
    return np.array(out)


def test_scores_brute_force_tiny():
    rng = np.random.default_rng(1)
    k = _bf16_values((12, 5), rng)
    q = _bf16_values((2, 3, 5), rng)
    got = O.window_scores(k, q, 0.37)
    np.testing.assert_allclose(got, _brute_scores(k, q, 0.37), rtol=1e-12, atol=1e-14)


def test_scores_invariant_total_mass():
    rng = np.random.default_rng(2)
    k = _bf16_values((200, 16), rng, 3.0)
    q = _bf16_values((4, 8, 16), rng)
    s = O.window_scores(k, q, 0.25, all_columns=True)
    assert abs(s.sum() - 4 * 8) < 1e-11
    assert np.all(s >= 0)


def test_scores_closed_form_uniform():
    # All logits equal: each window row j spreads mass 1 / (L - W + j + 1) over its visible keys.
    L, W, G, d = 50, 6, 3, 8
    k = np.zeros((L, d))
    q = np.ones((G, W, d))
    s = O.window_scores(k, q, 1.0)
    expect = G * sum(1.0 / (L - W + j + 1) for j in range(W))
    np.testing.assert_allclose(s, np.full(L - W, expect), rtol=1e-13)


def test_scores_single_row_is_softmax():
    rng = np.random.default_rng(3)
    L, d = 40, 16
    k = _bf16_values((L, d), rng)
    q = _bf16_values((1, 1, d), rng)
    s = O.window_scores(k, q, 0.2)
    ref = scipy.special.softmax(0.2 * (k @ q[0, 0]))
    np.testing.assert_allclose(s, ref[: L - 1], rtol=1e-12)


def test_scores_lse_matches_logsumexp():
    rng = np.random.default_rng(4)
    k = _bf16_values((30, 8), rng, 2.0)
    q = _bf16_values((2, 4, 8), rng)
    _, lse = O.window_scores(k, q, 0.5, return_lse=True)
    for h in range(2):
        for j in range(4):
            vis = 30 - 4 + j + 1
            ref = scipy.special.logsumexp(0.5 * (k[:vis] @ q[h, j]))
            assert abs(lse[h, j] - ref) < 1e-12


# ---------------------------------------------------------------- pooling and top-k
@pytest.mark.parametrize("kernel", [1, 3, 7, 15, 31])
def test_pool_matches_scipy_maximum_filter(kernel):
    rng = np.random.default_rng(5)
    x = rng.random(257)
    ref = scipy.ndimage.maximum_filter1d(x, size=kernel, mode="nearest")
    np.testing.assert_array_equal(O.pool_max(x, kernel), ref)


def test_pool_spike_closed_form():
    x = np.zeros(20)
    x[1] = 5.0
    p = O.pool_max(x, 7)
    assert list(np.nonzero(p)[0]) == [0, 1, 2, 3, 4]
    assert np.array_equal(O.pool_max(x, 1), x)


def test_topk_tie_break_lower_index():
    keys = np.array([1.0, 3.0, 2.0, 3.0, 2.0, 2.0, 0.5])
    assert list(O.topk_desc(keys, 4)) == [1, 3, 2, 4]
    rng = np.random.default_rng(6)
    keys = rng.integers(0, 5, 64).astype(np.float64)
    brute = sorted(range(64), key=lambda i: (-keys[i], i))[:17]
    assert list(O.topk_desc(keys, 17)) == brute


def test_snapkv_keep_all_and_window_last():
    rng = np.random.default_rng(7)
    L, W, d = 64, 8, 16
    k = _bf16_values((L, d), rng)
    v = _bf16_values((L, d), rng)
    q = _bf16_values((2, W, d), rng)
    kept, kk, vv, _, _ = O.snapkv_compress(k, v, q, keep=L, kernel=3, scale=0.25)
    assert np.array_equal(kept, np.arange(L))
    kept, kk, vv, score, pooled = O.snapkv_compress(k, v, q, keep=24, kernel=3, scale=0.25)
    assert len(kept) == 24
    assert np.array_equal(kept[-W:], np.arange(L - W, L))
    assert np.all(np.diff(kept) > 0)
    assert np.array_equal(kk, k[kept]) and np.array_equal(vv, v[kept])
    # every kept prefix token pools at least as high as every evicted one
    prefix = kept[:-W]
    evicted = np.setdiff1d(np.arange(L - W), prefix)
    assert pooled[prefix].min() >= pooled[evicted].max()


def test_snapkv_needle_recall_tiny_workload():
    """Sanity of the generator + oracle: planted needles survive a 256-token keep at 4K."""
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    wl = S.WORKLOADS["tiny_4k"]
    x = S.prefill_inputs(wl, seed=1001, device="cpu")
    L, W = wl.lens[0], wl.window
    for h in range(wl.n_kv):
        k = x["k"][0, h].double().numpy()
        v = x["v"][0, h].double().numpy()
        q = x["q_win"][0, h * wl.gqa:(h + 1) * wl.gqa].double().numpy()
        kept, *_ = O.snapkv_compress(k[:L], v[:L], q, keep=256, kernel=7, scale=O.default_scale(128))
        needles = set(x["needles"][0, h].tolist())
        assert needles <= set(kept.tolist())


# ---------------------------------------------------------------- summaries
def test_summaries_brute_force_and_partial_page():
    rng = np.random.default_rng(8)
    kc = _bf16_values((23, 6), rng)
    kmin, kmax = O.page_summaries(kc, 23, 4)
    assert kmin.shape == (6, 6)
    for pg in range(6):
        for c in range(6):
            vals = [kc[t, c] for t in range(pg * 4, min(23, pg * 4 + 4))]
            assert kmin[c, pg] == min(vals) and kmax[c, pg] == max(vals)
    a, b = O.page_summaries(kc, 23, 1)
    assert np.array_equal(a, kc.T) and np.array_equal(b, kc.T)


def test_append_matches_rebuild():
    rng = np.random.default_rng(9)
    cap, d, p = 40, 8, 4
    kc = np.zeros((cap, d))
    vc = np.zeros((cap, d))
    kc[:13] = _bf16_values((13, d), rng)
    kmin = np.zeros((d, 10))
    kmax = np.zeros((d, 10))
    a, b = O.page_summaries(kc, 13, p)
    kmin[:, :4], kmax[:, :4] = a, b
    length = 13
    for _ in range(9):
        length = O.append_token(kc, vc, length, kmin, kmax, _bf16_values(d, rng),
                                _bf16_values(d, rng), p)
    a, b = O.page_summaries(kc, length, p)
    P = a.shape[1]
    assert np.array_equal(kmin[:, :P], a) and np.array_equal(kmax[:, :P], b)


# ---------------------------------------------------------------- channel pick / approx / select
def test_channel_pick_known_answer_and_ties():
    q = np.zeros((2, 8))
    q[0] = [0.1, -3.0, 0.5, 0.0, 2.0, -0.25, 0.0, 1.0]
    q[1] = [0.1, 1.0, -0.5, 0.0, -2.0, 0.25, 0.0, 1.0]
    chosen, q_g = O.channel_pick(q, 3)
    # |q| sums: [0.2, 4, 1, 0, 4, 0.5, 0, 2] -> 1 and 4 (tie, both in), then 7
    assert list(chosen) == [1, 4, 7]
    np.testing.assert_array_equal(q_g, q.sum(axis=0))
    chosen, _ = O.channel_pick(q, 2)
    assert list(chosen) == [1, 4]
    q2 = np.ones((1, 4))
    assert list(O.channel_pick(q2, 2)[0]) == [0, 1]


def test_approx_upper_bound_all_channels():
    rng = np.random.default_rng(10)
    L, d, p = 64, 16, 4
    kc = _bf16_values((L, d), rng, 2.0)
    q = _bf16_values((4, d), rng)
    kmin, kmax = O.page_summaries(kc, L, p)
    chosen, q_g = O.channel_pick(q, d)
    A = O.approx_scores(q_g, chosen, kmin, kmax)
    true = kc @ q_g
    for pg in range(L // p):
        assert A[pg] >= true[pg * p:(pg + 1) * p].max() - 1e-12


def test_approx_page1_all_channels_is_exact_dot():
    rng = np.random.default_rng(11)
    kc = _bf16_values((30, 16), rng)
    q = _bf16_values((4, 16), rng)
    kmin, kmax = O.page_summaries(kc, 30, 1)
    chosen, q_g = O.channel_pick(q, 16)
    np.testing.assert_allclose(O.approx_scores(q_g, chosen, kmin, kmax), kc @ q_g, rtol=1e-12)


def test_approx_sign_choice():
    kmin = np.array([[-1.0, -2.0], [-3.0, -4.0]])
    kmax = np.array([[5.0, 6.0], [7.0, 8.0]])
    # q_g = [2, -1]: channel 0 reads Kmax (2*5, 2*6), channel 1 reads Kmin (-1*-3, -1*-4)
    A = O.approx_scores(np.array([2.0, -1.0]), np.array([0, 1]), kmin, kmax)
    np.testing.assert_array_equal(A, [13.0, 16.0])
    A = O.approx_scores(np.array([2.0, -1.0]), np.array([1]), kmin, kmax)
    np.testing.assert_array_equal(A, [3.0, 4.0])


def test_page_select_ties_and_order():
    s = np.array([1.0, 5.0, 5.0, 2.0, 5.0, 0.0])
    assert list(O.page_select(s, 2)) == [1, 2]
    assert list(O.page_select(s, 4)) == [1, 2, 3, 4]


# ---------------------------------------------------------------- attention and decode
def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(12)
    q = _bf16_values((4, 32), rng)
    k = _bf16_values((50, 32), rng)
    v = _bf16_values((50, 32), rng)
    got = O.attention(q, k, v, 0.3)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None, :], torch.from_numpy(k)[None, None].expand(1, 4, 50, 32),
        torch.from_numpy(v)[None, None].expand(1, 4, 50, 32), scale=0.3)[0, :, 0].numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_attention_closed_forms():
    rng = np.random.default_rng(13)
    q = _bf16_values((2, 8), rng)
    v = _bf16_values((5, 8), rng)
    k_same = np.tile(_bf16_values((1, 8), rng), (5, 1))
    np.testing.assert_allclose(O.attention(q, k_same, v, 1.0), np.tile(v.mean(0), (2, 1)),
                               rtol=1e-13)
    np.testing.assert_allclose(O.attention(q, k_same[:1], v[:1], 1.0), np.tile(v[0], (2, 1)))


def test_hybrid_budget_ge_len_is_dense():
    rng = np.random.default_rng(14)
    L, d = 100, 16
    kc = _bf16_values((L, d), rng)
    vc = _bf16_values((L, d), rng)
    q = _bf16_values((4, d), rng)
    kmin, kmax = O.page_summaries(kc, L, 4)
    r = O.hybrid_decode(q, kc, vc, L, kmin, kmax, budget=128, page=4, channels=4, scale=0.25)
    np.testing.assert_array_equal(r["out"], O.dense_decode(q, kc, vc, L, 0.25))


def test_hybrid_page1_all_channels_is_group_topk():
    rng = np.random.default_rng(15)
    L, d, B = 300, 16, 64
    kc = _bf16_values((L, d), rng)
    vc = _bf16_values((L, d), rng)
    q = _bf16_values((4, d), rng)
    kmin, kmax = O.page_summaries(kc, L, 1)
    r = O.hybrid_decode(q, kc, vc, L, kmin, kmax, budget=B, page=1, channels=d, scale=0.25)
    ref_out, ref_tokens = O.group_topk_attention(q, kc, vc, L, B // 2, 0.25)
    assert np.array_equal(r["tokens"], ref_tokens)
    np.testing.assert_allclose(r["out"], ref_out, rtol=1e-12)


def test_hybrid_token_count_is_half_budget():
    rng = np.random.default_rng(16)
    L, d, B, p = 1000, 32, 256, 4
    kc = _bf16_values((L, d), rng)
    vc = _bf16_values((L, d), rng)
    q = _bf16_values((4, d), rng)
    kmin, kmax = O.page_summaries(kc, L, p)
    r = O.hybrid_decode(q, kc, vc, L, kmin, kmax, budget=B, page=p, channels=8, scale=0.2)
    assert len(r["tokens"]) == B // 2
    assert len(r["pages"]) == B // 2 // p and len(r["channels"]) == 8
    # different queries select differently (selection is per step)
    q2 = _bf16_values((4, d), rng)
    r2 = O.hybrid_decode(q2, kc, vc, L, kmin, kmax, budget=B, page=p, channels=8, scale=0.2)
    assert not np.array_equal(r["pages"], r2["pages"])


# ---------------------------------------------------------------- RocketKV-MT (reading R17)
def test_mt_identity_kept_list_is_plain_decode():
    # keeping every token in order is RocketKV's decode on the full cache
    rng = np.random.default_rng(17)
    L, d, B, p = 700, 32, 128, 4
    kf = _bf16_values((L, d), rng)
    vf = _bf16_values((L, d), rng)
    q = _bf16_values((4, d), rng)
    kept = np.arange(L)
    kmin, kmax = O.mt_page_summaries(kf, kept, L, p)
    kmin0, kmax0 = O.page_summaries(kf, L, p)
    assert np.array_equal(kmin, kmin0) and np.array_equal(kmax, kmax0)
    r = O.mt_hybrid_decode(q, kf, vf, kept, L, kmin, kmax, B, p, 8, 0.2)
    r0 = O.hybrid_decode(q, kf, vf, L, kmin0, kmax0, B, p, 8, 0.2)
    assert np.array_equal(r["pages"], r0["pages"]) and np.array_equal(r["rows"], r0["tokens"])
    np.testing.assert_array_equal(r["out"], r0["out"])


def test_mt_evicted_rows_never_matter():
    # "SCBench Results": RocketKV-MT keeps every token in memory, yet the decode picks only from
    # the filtered ones, so rows outside the kept list may hold anything without changing a step
    rng = np.random.default_rng(18)
    L, d, B, p, n_kept = 2000, 32, 128, 4, 500
    kf = _bf16_values((L, d), rng)
    vf = _bf16_values((L, d), rng)
    q = _bf16_values((4, d), rng)
    kept = np.sort(rng.choice(L, n_kept, replace=False))
    kmin, kmax = O.mt_page_summaries(kf, kept, n_kept, p)
    r = O.mt_hybrid_decode(q, kf, vf, kept, n_kept, kmin, kmax, B, p, 8, 0.2)
    assert set(r["rows"].tolist()) <= set(kept.tolist())
    assert len(r["rows"]) == B // 2
    others = np.setdiff1d(np.arange(L), kept)
    kf2, vf2 = kf.copy(), vf.copy()
    kf2[others] = 1e3 * _bf16_values((len(others), d), rng)
    vf2[others] = -7.0
    kmin2, kmax2 = O.mt_page_summaries(kf2, kept, n_kept, p)
    r2 = O.mt_hybrid_decode(q, kf2, vf2, kept, n_kept, kmin2, kmax2, B, p, 8, 0.2)
    assert np.array_equal(r["rows"], r2["rows"])
    np.testing.assert_array_equal(r["out"], r2["out"])


def test_mt_append_matches_rebuild():
    # generated tokens go to the end of the full cache and of the kept sequence; the summaries
    # kept incrementally equal those rebuilt from the final kept sequence
    rng = np.random.default_rng(19)
    L, d, p, n_kept, steps, cap = 600, 16, 4, 101, 9, 640
    kf = np.zeros((cap, d))
    vf = np.zeros((cap, d))
    kf[:L] = _bf16_values((L, d), rng)
    vf[:L] = _bf16_values((L, d), rng)
    kept = np.full(n_kept + steps, -1)
    kept[:n_kept] = np.sort(rng.choice(L, n_kept, replace=False))
    P_cap = (n_kept + steps + p - 1) // p
    kmin = np.zeros((d, P_cap))
    kmax = np.zeros((d, P_cap))
    a, b = O.mt_page_summaries(kf, kept, n_kept, p)
    kmin[:, :a.shape[1]], kmax[:, :a.shape[1]] = a, b
    full_len, nk = L, n_kept
    new = []
    for _ in range(steps):
        nkv = _bf16_values((2, d), rng)
        new.append(nkv)
        full_len, nk = O.mt_append_token(kf, vf, full_len, kept, nk, kmin, kmax, nkv[0], nkv[1], p)
    assert (full_len, nk) == (L + steps, n_kept + steps)
    assert np.array_equal(kept[n_kept:], np.arange(L, L + steps))
    assert np.array_equal(kf[L:L + steps], np.stack([x[0] for x in new]))
    ra, rb = O.mt_page_summaries(kf, kept, nk, p)
    P = (nk + p - 1) // p
    assert np.array_equal(kmin[:, :P], ra) and np.array_equal(kmax[:, :P], rb)


# ---------------------------------------------------------------- even-split planner (R18)
def test_plan_even_split_worked_example():
    g = _golden("planner_worked_example.json")
    keep, page, channels, _ = O.plan_even_split(g["ctx"], g["budget"], g["head_dim"])
    assert page == g["page"]
    assert g["head_dim"] // channels == g["head_dim_ratio"]
    assert g["ctx"] // keep == g["per_stage_ratio"]


@pytest.mark.parametrize("ctx,budget", [(131072, 512), (32768, 256), (65536, 512), (1 << 20, 64),
                                        (8192, 1024), (100, 256), (4096, 4096), (131072, 64)])
def test_plan_even_split_identities(ctx, budget):
    d = 128
    keep, page, channels, _ = O.plan_even_split(ctx, budget, d)
    ratio = ctx / budget
    assert page & (page - 1) == 0 and 1 <= page <= min(64, budget // 2)
    assert 1 <= channels <= d
    assert keep == min(ctx, budget * page * d // channels)
    if ratio > 1 and page < min(64, budget // 2):
        # the page is the power of two nearest R^(1/4) (log2 scale), unless clamped
        assert abs(math.log2(page) - math.log2(ratio) / 4) <= 0.5 + 1e-12
    if 1 < channels < d:
        # page * d / channels approximates the stage-2 ratio sqrt(R) up to channel rounding
        assert abs(d * page / channels - math.sqrt(ratio)) <= d * page / channels / (2 * channels - 1) + 1e-9
    if ratio >= 1 and math.log2(ratio) % 4 == 0 and page < min(64, budget // 2):
        # ratios 16^k split exactly: page = d / channels = R^(1/4)
        assert page == round(ratio ** 0.25) and d // channels == page


# ---------------------------------------------------------------- SnapKV without the GQA sum (R19)
def test_per_head_scores_sum_to_group_scores():
    rng = np.random.default_rng(20)
    L, W, G, d = 300, 8, 4, 16
    k = _bf16_values((L, d), rng)
    q = _bf16_values((G, W, d), rng)
    group = O.window_scores(k, q, 0.25)
    per_head = [O.window_scores(k, q[h:h + 1], 0.25) for h in range(G)]
    np.testing.assert_allclose(np.sum(per_head, axis=0), group, rtol=1e-12)
    res = O.snapkv_compress_per_head(k, _bf16_values((L, d), rng), q, 64, 7, 0.25)
    assert len(res) == G
    for h, (kept, kc, _, score, _) in enumerate(res):
        np.testing.assert_array_equal(score, per_head[h])
        assert np.array_equal(kept[-W:], np.arange(L - W, L)) and np.array_equal(kc, k[kept])
    # heads that look at different parts of the prompt keep different tokens
    assert not all(np.array_equal(res[0][0], r[0]) for r in res[1:])


# ---------------------------------------------------------------- paged cache (R20)
def test_paged_round_trip_and_decode():
    rng = np.random.default_rng(21)
    L, d, n_kv, block, B, p = 700, 16, 2, 64, 128, 4
    kc = _bf16_values((n_kv, L, d), rng)
    vc = _bf16_values((n_kv, L, d), rng)
    nb = (L + block - 1) // block
    table = rng.permutation(3 * nb)[:nb]              # scattered, non-contiguous blocks
    kp = np.full((3 * nb, n_kv, block, d), np.nan)
    vp = np.full_like(kp, np.nan)
    for g in range(n_kv):
        O.paged_scatter(kp, table, kc[g], g)
        O.paged_scatter(vp, table, vc[g], g)
        assert np.array_equal(O.paged_view(kp, table, L, g), kc[g])
    # token 65 with blocks of 64 is row 1 of the table's second block; token 699 row 59 of the
    # eleventh
    assert np.array_equal(kp[table[1], 1, 1], kc[1, 65])
    assert np.array_equal(kp[table[10], 0, 59], kc[0, 699])
    q = _bf16_values((4, d), rng)
    kv0 = O.paged_view(kp, table, L, 1)
    kmin, kmax = O.page_summaries(kv0, L, p)
    r = O.hybrid_decode(q, kv0, O.paged_view(vp, table, L, 1), L, kmin, kmax, B, p, 8, 0.2)
    k1min, k1max = O.page_summaries(kc[1], L, p)
    r1 = O.hybrid_decode(q, kc[1], vc[1], L, k1min, k1max, B, p, 8, 0.2)
    assert np.array_equal(r["tokens"], r1["tokens"])
    np.testing.assert_array_equal(r["out"], r1["out"])


# ---------------------------------------------------------------- average pooling (R21)
def test_pool_avg_hand_example_and_invariants():
    x = np.array([4.0, 0.0, 2.0, 8.0, 1.0])
    # kernel 3: clipped windows [4,0], [4,0,2], [0,2,8], [2,8,1], [8,1]
    np.testing.assert_allclose(O.pool_avg(x, 3), [2.0, 2.0, 10 / 3, 11 / 3, 4.5], rtol=1e-15)
    np.testing.assert_array_equal(O.pool_avg(x, 1), x)
    rng = np.random.default_rng(22)
    y = rng.random(200)
    for kern in (3, 7, 15, 31):
        a = O.pool_avg(y, kern)
        assert np.all(a <= O.pool_max(y, kern) + 1e-15)
        assert np.allclose(O.pool_avg(np.full(50, 0.25), kern), 0.25)
        # interior positions are the plain moving average
        r = kern // 2
        np.testing.assert_allclose(a[r:-r], np.convolve(y, np.ones(kern) / kern, mode="valid"),
                                   rtol=1e-12)


# ---------------------------------------------------------------- RocketKV-MT across turns (R22)
def test_mt_second_turn_recovers_tokens_the_first_evicted():
    # "SCBench Results": tokens that the first turn's filtering drops can matter to a later turn,
    # and RocketKV-MT, which evicts nothing, finds them again when it filters the full history.
    # Keys that only the second turn's queries single out are planted in the first prompt.
    from sparse_kv_cache_snapkv_gb300 import synthetic as S
    wl = S.Workload("mt2", 1, 1, 2, 4, 128, (6000,), 32, 256, needles=8)
    x = S.prefill_inputs(wl, seed=1)
    t2 = S.second_turn_inputs(wl, x, 256, 8, seed=101)
    nk, nv = S.append_tokens(wl, 16, x["sigma"], seed=201)
    keep, scale = 1024, 1 / math.sqrt(128)
    for h in range(2):
        k = x["k"][0, h].double().numpy()
        kept1 = O.snapkv_compress(k, k, x["q_win"][0, 4 * h:4 * h + 4].double().numpy(), keep,
                                  7, scale)[0]
        hist = np.concatenate([k, nk[:, 0, h].double().numpy(),
                               t2["new_k"][0, h].double().numpy()])
        L2 = hist.shape[0]
        q2 = t2["q_win"][0, 4 * h:4 * h + 4].double().numpy()
        kept2 = O.mt_refilter(hist, L2, q2, keep, 7, scale)
        n2 = t2["needles"][0, h].numpy()
        assert np.isin(n2, kept1).sum() <= 2            # the first turn drops them
        assert np.isin(n2, kept2).all()                 # the second finds them again
        assert np.array_equal(kept2[-32:], np.arange(L2 - 32, L2))
        # the re-filter is SnapKV++ on the history: with the history equal to the first prompt
        # and the first turn's queries it returns the first turn's list
        assert np.array_equal(O.mt_refilter(k, 6000, x["q_win"][0, 4 * h:4 * h + 4].double()
                                            .numpy(), keep, 7, scale), kept1)
        # rows past full_len are not part of the history
        padded = np.concatenate([hist, np.full((50, 128), 1e3)])
        assert np.array_equal(O.mt_refilter(padded, L2, q2, keep, 7, scale), kept2)
