"""Plain fp64 CPU oracle for the RocketKV hot path (SnapKV++ eviction + hybrid sparse decode).

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module: only the tests,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``
call it. It shares no code with the CUDA library and never imports it.

Every function takes float64 numpy arrays that hold the exact values of the bf16 inputs and
computes in float64. It is deliberately slow and literal: each step follows the method's text in
the order the pages give it, with numpy library primitives (matmul, exp, sort) as the only
building blocks.

Sources (the pages, cited by title and section):
  [P1] "RocketKV: Accelerating Long-Context LLM Inference via Two-Stage KV Cache Compression",
       summarizepaper.com summary of arXiv 2502.14051v1 -- "Key points", "Summary".
  [P3] the same title on paperhub.cn (OpenReview author responses) -- paragraphs
       "Novelty: RocketKV is SnapKV + QUEST", "Potential Sensitivity to Kernel Size in SnapKV++",
       "Lack of Direct Latency Comparison", "Is Needle Among Evicted Tokens",
       "Explanation of Calculating Approximate Attention Scores", "Measurement of Exact-TopK",
       "Are Different KV Tokens Retrieved at Each Decoding Step?",
       "Is Page Always Divided Into 4?", "Novelty of SnapKV++".
  [P4] the same title on pith.science (abstract v3).

Readings taken where the pages leave a step open (each restated at its function):
  R1  stage-1 keep N1 = min(L, B * p * d / c) (the 128K / 512 worked example in
      "Is Page Always Divided Into 4?" gives 8192 = 16 * 512 with p = 4, c = d / 4).
  R2  stage-1 scores are softmax probabilities (logits scaled by `scale`, normalised over every key
      visible to that window query: the prefix plus the causal part of the window), summed over the
      window rows and over the query heads of the KV head's group. Only prefix columns are ranked;
      the window tokens are always kept.
  R3  adaptive pooling kernel: L <= 8192 -> 7, L <= 32768 -> 15, else 31 (the pages only say
      that longer contexts get larger kernels).
  R4  max pooling, stride 1, same length, window clipped at both ends.
  R5  top-k order: larger key first, equal keys -> lower index. Kept indices stored ascending, then
      the window positions.
  R6  N1 >= L keeps everything; a cache of len <= B is attended densely (no approximation).
  R7  channel pick on sum_h |q_h|; score and Kmin/Kmax sign choice on q_g = sum_h q_h.
  R8  q_g[i] >= 0 reads Kmax (the product is 0 at q_g[i] == 0 either way).
  R9  approximate scores are unscaled.
  R10 S = floor((B/2) / p) whole pages are selected; a partial last page counts its valid tokens.
  R11 the summary of a partial last page is over its valid tokens only.
  R12 decode appends (when given) happen before attending; the new token is selectable.
  R13 attention scale as given (1/sqrt(d) by default); output kept in float64.
  (R14-R16 concern the seeded synthetic inputs, not this module.)
  R18 the even split of "Is Page Always Divided Into 4?" for any ratio R = ctx / B: sqrt(R) per
      stage, stage 2's share split evenly between page size and channel reduction; the page is the
      power of two nearest R^(1/4) on a log2 scale (halves round up) within [1, min(64, B/2)],
      channels = round(d * page / sqrt(R)) within [1, d], keep as in R1.
  R21 average pooling (an ablation variant; the pages describe max pooling only): the mean over
      the in-range positions of the clipped window.
  R20 a paged (block-table) compact cache is a storage layout only: every step computes on the
      rows the table names, in token order, exactly as on the contiguous cache.
  R19 SnapKV without the GQA enhancement ([P1] "Key points": the ablation against plain SnapKV):
      each query head scores with its own W window rows only, and keeps its own top-k.
  R17 RocketKV-MT ([P3] "SCBench Results"): nothing is evicted; the decode runs the stage-2 steps
      on the sequence of kept tokens (stage 1's kept positions in its order, then the tokens
      generated since), whose rows stay in the full cache. The pages do not say where generated
      tokens go; they are appended to the full cache and to the kept sequence, and are selectable
      (as in R12).
  R22 RocketKV-MT across turns ([P3] "SCBench Results": the next turn's prefill takes every
      earlier token as its prefix and SnapKV++ filters the unfiltered history again): a later
      turn's history is the full cache in row order (earlier prompts, generated tokens, the new
      input), its window is the last W queries of the new input, and the new kept list replaces
      the old one; the turn's generated tokens are appended to it as in R17.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "plan", "adaptive_kernel_size", "window_scores", "pool_max", "pool_avg", "topk_desc",
    "snapkv_compress", "page_summaries", "channel_pick", "approx_scores", "page_select",
    "attention", "dense_decode", "hybrid_decode", "group_topk_attention", "append_token",
    "kept_view", "mt_page_summaries", "mt_hybrid_decode", "mt_append_token", "mt_refilter",
    "plan_even_split", "snapkv_compress_per_head", "paged_view", "paged_scatter",
]


# --------------------------------------------------------------------------------------------
# Planning: the compression-ratio decomposition
# --------------------------------------------------------------------------------------------
def adaptive_kernel_size(ctx: int) -> int:
    """Pooling kernel from the prompt length (reading R3).

    [P3] "Potential Sensitivity to Kernel Size in SnapKV++": the kernel size is chosen from the
    sequence length, larger for longer inputs; [P1] "Key points" ties kernel size to sequence
    length. The table itself is not on the pages: 7 up to 8K tokens, 15 up to 32K, 31 beyond.
    """
    if ctx <= 8192:
        return 7
    if ctx <= 32768:
        return 15
    return 31


def plan(ctx: int, budget: int, head_dim: int, page: int = 0, channels: int = 0):
    """Resolve (keep N1, page size p, channels c, pooling kernel) for one sequence.

    [P3] "Is Page Always Divided Into 4?": the overall ratio ctx/B is split evenly between the two
    stages, and the second stage's share evenly between the sequence dimension (page size) and the
    head dimension (channels kept); 128K / 512 -> 256x -> 16x per stage -> page 4 and 4x fewer
    channels. [P3] "Novelty: RocketKV is SnapKV + QUEST": ratio 16 split as 4 x 4.
    Reading R1: p defaults to 4 and c to d/4, and N1 = min(ctx, B * p * d / c), so that the
    approximation step reads exactly as many bytes as B/2 tokens of K and V.
    """
    if page == 0:
        page = 4
    if channels == 0:
        channels = head_dim // 4
    keep = min(ctx, budget * page * head_dim // channels)
    return keep, page, channels, adaptive_kernel_size(ctx)


def plan_even_split(ctx: int, budget: int, head_dim: int):
    """(keep, page, channels, kernel) from the even split of the ratio (reading R18).

    [P3] "Is Page Always Divided Into 4?": ctx / B is split evenly between the two stages and
    stage 2's share evenly between the sequence and head dimensions; the page size "can vary for
    other compression ratios".
    """
    ratio = ctx / budget
    stage2 = math.sqrt(ratio)
    steps = math.floor(math.log2(stage2) / 2.0 + 0.5) if stage2 > 0 else 0
    page = 1
    for _ in range(max(0, steps)):
        if page >= 64 or page * 2 > budget // 2:
            break
        page *= 2
    channels = min(head_dim, max(1, round(head_dim * page / stage2)))
    keep = min(ctx, budget * page * head_dim // channels)
    return keep, page, channels, adaptive_kernel_size(ctx)


# --------------------------------------------------------------------------------------------
# Stage 1: SnapKV++ eviction
# --------------------------------------------------------------------------------------------
def window_scores(k: np.ndarray, q_win: np.ndarray, scale: float, return_lse: bool = False,
                  all_columns: bool = False):
    """Observation-window scores of the prefix, summed over the window and the GQA group.

    k: [L, d] keys of one (sequence, layer, KV head); q_win: [G, W, d], the last W queries of the
    G query heads that share this KV head. Window row j sits at absolute position L - W + j and
    sees keys 0 .. L - W + j. Returns score[i] for the L - W prefix positions (reading R2):
        score[i] = sum_h sum_j softmax_row(h, j)[i]
    (all L column sums when `all_columns`; those add up to G * W).
    [P1] "Key points" (SnapKV with the grouped-query enhancement); [P3] "Novelty of SnapKV++"
    (the enhancement scores each KV head once from its whole group).
    """
    L, d = k.shape
    G, W, _ = q_win.shape
    rows = q_win.reshape(G * W, d)
    logits = (rows @ k.T) * scale                      # [G*W, L]
    pos = (L - W) + np.tile(np.arange(W), G)           # absolute position of each row
    visible = np.arange(L)[None, :] <= pos[:, None]
    logits = np.where(visible, logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    denom = e.sum(axis=1, keepdims=True)
    probs = e / denom
    score = probs.sum(axis=0) if all_columns else probs[:, : L - W].sum(axis=0)
    if return_lse:
        return score, (m[:, 0] + np.log(denom[:, 0])).reshape(G, W)
    return score


def pool_max(x: np.ndarray, kernel: int) -> np.ndarray:
    """1-D max pooling, stride 1, same length, window clipped at the ends (reading R4).

    [P3] "Potential Sensitivity to Kernel Size in SnapKV++" (pooling with an adaptive size).
    """
    assert kernel % 2 == 1 and kernel >= 1
    r = kernel // 2
    n = x.shape[0]
    out = np.empty_like(x)
    for i in range(n):
        out[i] = x[max(0, i - r): min(n, i + r + 1)].max()
    return out


def pool_avg(x: np.ndarray, kernel: int) -> np.ndarray:
    """1-D average pooling, stride 1, same length: the mean over the in-range positions of the
    window (reading R21; the pages describe max pooling only, this is the ablation variant)."""
    assert kernel % 2 == 1 and kernel >= 1
    r = kernel // 2
    n = x.shape[0]
    out = np.empty_like(x)
    for i in range(n):
        out[i] = x[max(0, i - r): min(n, i + r + 1)].mean()
    return out


def topk_desc(keys: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest keys; equal keys -> lower index first (reading R5).

    Returned in selection order (largest first). A full stable sort, nothing clever.
    """
    idx = np.arange(keys.shape[0])
    order = np.lexsort((idx, -keys))                    # primary: -key, secondary: index
    return order[:k]


def snapkv_compress(k: np.ndarray, v: np.ndarray, q_win: np.ndarray, keep: int, kernel: int,
                    scale: float, pooling: str = "max"):
    """SnapKV++ for one (sequence, layer, KV head): score, pool, top-k, gather.

    [P3] "Is Needle Among Evicted Tokens": eviction is independent per head and per layer.
    [P3] "Measurement of Exact-TopK": SnapKV prunes the prompt by a one-time top-k filter.
    Returns (kept_idx ascending prefix then window, K_kept, V_kept, prefix scores, pooled scores).
    Reading R6: keep >= L keeps every token (scores are still returned).
    """
    L = k.shape[0]
    W = q_win.shape[1]
    score = window_scores(k, q_win, scale)
    pooled = pool_avg(score, kernel) if pooling == "avg" else pool_max(score, kernel)
    if keep >= L:
        kept = np.arange(L)
    else:
        prefix = np.sort(topk_desc(pooled, keep - W))
        kept = np.concatenate([prefix, np.arange(L - W, L)])
    return kept, k[kept], v[kept], score, pooled


def snapkv_compress_per_head(k: np.ndarray, v: np.ndarray, q_win: np.ndarray, keep: int,
                             kernel: int, scale: float):
    """SnapKV without the GQA enhancement (reading R19): `snapkv_compress` run for each query head
    of the group alone (its W window rows), each keeping its own rows of the shared K/V head.
    q_win: [G, W, d]. Returns one snapkv_compress result per query head.
    """
    return [snapkv_compress(k, v, q_win[h:h + 1], keep, kernel, scale)
            for h in range(q_win.shape[0])]


# --------------------------------------------------------------------------------------------
# Stage 2: hybrid sparse decode attention
# --------------------------------------------------------------------------------------------

def page_summaries(kc: np.ndarray, length: int, page: int):
    """Element-wise Kmin / Kmax per page of consecutive tokens, channel-major [d, P].

    [P3] "Explanation of Calculating Approximate Attention Scores": K is split into pages of
    consecutive tokens and each page records its element-wise min and max. Reading R11: the last
    page covers only its valid tokens.
    """
    d = kc.shape[1]
    P = (length + page - 1) // page
    kmin = np.empty((d, P))
    kmax = np.empty((d, P))
    for pg in range(P):
        rows = kc[pg * page: min(length, (pg + 1) * page)]
        kmin[:, pg] = rows.min(axis=0)
        kmax[:, pg] = rows.max(axis=0)
    return kmin, kmax


def channel_pick(q: np.ndarray, channels: int):
    """Top-|q| channels of a GQA group; returns (channels ascending, q_g = sum_h q_h).

    [P3] "Explanation of Calculating Approximate Attention Scores": only head-dim positions where
    |q| is large are used, and for GQA the selection uses the group sum of q or |q| so that all
    heads of a group select alike. Reading R7: |q| summed for the pick, signed q for the score.
    """
    mag = np.abs(q).sum(axis=0)
    chosen = np.sort(topk_desc(mag, channels))
    return chosen, q.sum(axis=0)


def approx_scores(q_g: np.ndarray, chosen: np.ndarray, kmin: np.ndarray, kmax: np.ndarray):
    """Approximate page score: sum over the kept channels of max(q*Kmin, q*Kmax).

    [P3] "Explanation of Calculating Approximate Attention Scores": per page, max(q x Kmin,
    q x Kmax) bounds the highest score inside the page, and only one of Kmin / Kmax is fetched per
    position, chosen by the sign of q. Reading R8 (q >= 0 -> Kmax), R9 (unscaled).
    """
    P = kmin.shape[1]
    total = np.zeros(P)
    for i in chosen:
        row = kmax[i] if q_g[i] >= 0 else kmin[i]
        total += q_g[i] * row
    return total


def page_select(scores: np.ndarray, n_select: int) -> np.ndarray:
    """The n_select pages with the highest approximate score, ascending (reading R5, R10).

    [P3] "Explanation of Calculating Approximate Attention Scores": "select pages with higher
    scores".
    """
    return np.sort(topk_desc(scores, min(n_select, scores.shape[0])))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of G query heads [G, d] over T tokens k, v [T, d] -> [G, d]."""
    logits = (q @ k.T) * scale
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    return (e / e.sum(axis=1, keepdims=True)) @ v


def dense_decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, length: int, scale: float):
    """Full-KV decode attention, the baseline the pages compare against ([P1] "Key points")."""
    return attention(q, k[:length], v[:length], scale)


def hybrid_decode(q: np.ndarray, kc: np.ndarray, vc: np.ndarray, length: int,
                  kmin: np.ndarray, kmax: np.ndarray, budget: int, page: int, channels: int,
                  scale: float):
    """One hybrid decode step for one (sequence, layer, KV head) and its G query heads.

    [P3] "Lack of Direct Latency Comparison": half the token budget is spent on the approximation
    (steps 1, 2) and half on sparse attention (step 3). [P3] "Explanation of Calculating
    Approximate Attention Scores": steps 1-2 (channel pick, approximate score, page select).
    [P3] "Are Different KV Tokens Retrieved at Each Decoding Step?": the selection is redone per
    step. Reading R6: length <= budget attends densely over every token.
    Returns a dict with out [G, d], chosen channels, approx scores, selected pages, token ids.
    """
    if length <= budget:
        tokens = np.arange(length)
        return {"out": attention(q, kc[tokens], vc[tokens], scale), "tokens": tokens,
                "channels": None, "scores": None, "pages": None}
    chosen, q_g = channel_pick(q, channels)
    P = (length + page - 1) // page
    scores = approx_scores(q_g, chosen, kmin[:, :P], kmax[:, :P])
    pages = page_select(scores, (budget // 2) // page)
    tokens = np.concatenate([np.arange(pg * page, min(length, (pg + 1) * page)) for pg in pages])
    return {"out": attention(q, kc[tokens], vc[tokens], scale), "tokens": tokens,
            "channels": chosen, "scores": scores, "pages": pages}


def group_topk_attention(q: np.ndarray, kc: np.ndarray, vc: np.ndarray, length: int, k: int,
                         scale: float):
    """Exact top-k attention shared by a GQA group: rank tokens by the true group logit sum.

    [P3] "Measurement of Exact-TopK": the oracle top-k scheme picks the top-k tokens by their true
    scores at every step. With the selection shared per group ([P3] "Explanation of Calculating
    Approximate Attention Scores"), the true group score of token t is sum_h q_h . k_t.
    Written independently of `hybrid_decode`: it is what that function must reduce to with page
    size 1 and all channels kept.
    """
    true_scores = kc[:length] @ q.sum(axis=0)
    tokens = np.sort(topk_desc(true_scores, min(k, length)))
    return attention(q, kc[tokens], vc[tokens], scale), tokens


def append_token(kc: np.ndarray, vc: np.ndarray, length: int, kmin: np.ndarray,
                 kmax: np.ndarray, new_k: np.ndarray, new_v: np.ndarray, page: int):
    """Append one decode token and update the page it lands in (reading R12, R11).

    Arrays are modified in place; returns the new length. A token that opens a page sets that
    page's Kmin = Kmax = new_k; otherwise the page's min / max absorb it.
    """
    kc[length] = new_k
    vc[length] = new_v
    pg = length // page
    if length % page == 0:
        kmin[:, pg] = new_k
        kmax[:, pg] = new_k
    else:
        kmin[:, pg] = np.minimum(kmin[:, pg], new_k)
        kmax[:, pg] = np.maximum(kmax[:, pg], new_k)
    return length + 1


# --------------------------------------------------------------------------------------------
# RocketKV-MT: the full cache is kept, the decode sees only the kept tokens (reading R17)
# --------------------------------------------------------------------------------------------
def kept_view(full: np.ndarray, kept: np.ndarray, n_kept: int) -> np.ndarray:
    """Rows of the kept sequence: full[kept[j]] for j < n_kept, in kept-list order.

    [P3] "SCBench Results": in RocketKV-MT all input tokens stay in memory and the hybrid
    attention selects only among the tokens SnapKV++ identified as important.
    """
    return full[np.asarray(kept[:n_kept], dtype=np.int64)]


def mt_page_summaries(k_full: np.ndarray, kept: np.ndarray, n_kept: int, page: int):
    """Kmin / Kmax over pages of the kept sequence (R17, then R11)."""
    return page_summaries(kept_view(k_full, kept, n_kept), n_kept, page)


def mt_hybrid_decode(q: np.ndarray, k_full: np.ndarray, v_full: np.ndarray, kept: np.ndarray,
                     n_kept: int, kmin: np.ndarray, kmax: np.ndarray, budget: int, page: int,
                     channels: int, scale: float):
    """One RocketKV-MT decode step: `hybrid_decode` on the kept sequence (R17).

    Pages and token ids in the result count positions of the kept sequence; "rows" gives the
    attended rows of the full cache.
    """
    kc = kept_view(k_full, kept, n_kept)
    vc = kept_view(v_full, kept, n_kept)
    r = hybrid_decode(q, kc, vc, n_kept, kmin, kmax, budget, page, channels, scale)
    r["rows"] = np.asarray(kept[:n_kept], dtype=np.int64)[r["tokens"]]
    return r


def mt_append_token(k_full: np.ndarray, v_full: np.ndarray, full_len: int, kept: np.ndarray,
                    n_kept: int, kmin: np.ndarray, kmax: np.ndarray, new_k: np.ndarray,
                    new_v: np.ndarray, page: int):
    """Append one generated token in RocketKV-MT (R17): it takes row full_len of the full cache
    and position n_kept of the kept sequence, whose page summary absorbs it as in
    `append_token`. Arrays are modified in place; returns (full_len + 1, n_kept + 1).
    """
    k_full[full_len] = new_k
    v_full[full_len] = new_v
    kept[n_kept] = full_len
    pg = n_kept // page
    if n_kept % page == 0:
        kmin[:, pg] = new_k
        kmax[:, pg] = new_k
    else:
        kmin[:, pg] = np.minimum(kmin[:, pg], new_k)
        kmax[:, pg] = np.maximum(kmax[:, pg], new_k)
    return full_len + 1, n_kept + 1


def mt_refilter(k_full: np.ndarray, full_len: int, q_win: np.ndarray, keep: int, kernel: int,
                scale: float) -> np.ndarray:
    """The kept list of a later RocketKV-MT turn (R22): SnapKV++ over the whole history
    k_full[:full_len] with this turn's window queries. Returns the kept positions (ascending
    prefix, then the window), which index the full cache directly.
    [P3] "SCBench Results".
    """
    hist = k_full[:full_len]
    return snapkv_compress(hist, hist, q_win, keep, kernel, scale)[0]


# --------------------------------------------------------------------------------------------
# Paged compact cache (reading R20)
# --------------------------------------------------------------------------------------------
def paged_view(pool: np.ndarray, table: np.ndarray, n_tok: int, g: int) -> np.ndarray:
    """Rows of tokens 0 .. n_tok-1 of K/V head g from a pool [blocks][n_kv][block][d] whose token
    t sits in block table[t // block], row t % block."""
    block = pool.shape[2]
    t = np.arange(n_tok)
    return pool[np.asarray(table, dtype=np.int64)[t // block], g, t % block]


def paged_scatter(pool: np.ndarray, table: np.ndarray, rows: np.ndarray, g: int) -> None:
    """Write rows (token order) of K/V head g into their blocks (in place)."""
    block = pool.shape[2]
    t = np.arange(rows.shape[0])
    pool[np.asarray(table, dtype=np.int64)[t // block], g, t % block] = rows


def default_scale(head_dim: int) -> float:
    """1 / sqrt(d) (reading R13)."""
    return 1.0 / math.sqrt(head_dim)
