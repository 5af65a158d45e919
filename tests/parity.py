"""GPU-vs-oracle acceptance rules shared by the parity tests.

* Index sets (kept tokens, channels, pages): equal to the oracle's, except that elements whose
  oracle key lies within the tie band around the k-th key, |s_i - s_k| <= 1e-4 * |s_k|, may be
  exchanged for one another.
* Approximate page scores: |gpu - ref| <= 2 gamma(c + 9) * sum_{i in C} |q_g[i] * K_sel[i][pg]|,
  gamma(n) = n u32 / (1 - n u32), u32 = 2^-24: the kernel forms q_g as an fp32 sum of at most 8
  bf16 query values and the score as fp32 fused multiply-adds over the c kept channels plus one
  addition joining two partial sums, so at most c + 9 roundings of fp32, each bounded by u32
  times the magnitude (the standard bound for a sum in any order); doubled.
* Attention outputs (bf16), per query head h and channel c: |gpu - ref| <= 2^-7 * (spread + |ref|)
  + 1e-5, ref = the oracle's attention in float64 over the tokens the kernel attended (the GPU's
  own selection when that differs from the oracle's inside the tie band). The kernel rounds each
  probability it feeds to P.V to bf16 (round to nearest, relative error at most u = 2^-8 for an
  8-bit significand) and sums the normaliser from the same rounded values, so its output moves
  by sum_t p_t eps_t (v_t[c] - ref[c]), at most u * spread with spread = sum_t p_t |v_t[c] -
  ref[c]|; the output's own rounding to bf16 adds u * |ref|. The bound is doubled for the fp32
  logits and accumulations, and 1e-5 covers values near zero.
"""
import numpy as np

from oracle import rocketkv as O

BAND_REL = 1e-4
OUT_ABS = 2e-3
OUT_REL = 1e-2


def check_selection(gpu_sel, keys, k, what="selection"):
    """gpu_sel: selected indices (any order); keys: oracle fp64 keys; k: number selected."""
    gpu = np.sort(np.asarray(gpu_sel, dtype=np.int64))
    assert gpu.shape[0] == k, f"{what}: {gpu.shape[0]} selected, expected {k}"
    assert np.unique(gpu).shape[0] == k, f"{what}: duplicate indices"
    assert gpu.min() >= 0 and gpu.max() < keys.shape[0], f"{what}: index out of range"
    order = np.lexsort((np.arange(keys.shape[0]), -keys))
    ref = np.sort(order[:k])
    if np.array_equal(gpu, ref):
        return 0
    sk = keys[order[k - 1]]
    band = BAND_REL * abs(sk)
    must = np.nonzero(keys > sk + band)[0]
    never = np.nonzero(keys < sk - band)[0]
    gset = set(gpu.tolist())
    missing = [i for i in must if i not in gset]
    extra = [i for i in never if i in gset]
    assert not missing and not extra, (
        f"{what}: outside the tie band: missing {missing[:8]} (keys {keys[missing[:8]]}), "
        f"extra {extra[:8]} (keys {keys[extra[:8]]}), k-th key {sk}")
    return len(set(ref.tolist()) ^ gset) // 2


BF16_REL = 2.0 ** -8  # unit roundoff of bf16 round-to-nearest (8-bit significand)


def attention_tolerance(q, k, v, scale, ref):
    """Per (query head, channel): 2 * 2^-8 * (sum_t p_t |v_t - ref| + |ref|) + 1e-5, with p the
    softmax probabilities of q over the attended keys (the rounding model above)."""
    logits = (np.asarray(q, dtype=np.float64) @ np.asarray(k, dtype=np.float64).T) * scale
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    v = np.asarray(v, dtype=np.float64)
    spread = np.stack([p[h] @ np.abs(v - ref[h]) for h in range(p.shape[0])])
    return 2.0 * BF16_REL * (spread + np.abs(ref)) + 1e-5


def check_attention(gpu_out, q, k, v, scale, what="output"):
    """gpu_out [G, d] against the oracle's attention of q [G, d] over the attended k, v [T, d]."""
    ref = O.attention(q, k, v, scale)
    gpu = np.asarray(gpu_out, dtype=np.float64)
    err = np.abs(gpu - ref)
    tol = attention_tolerance(q, k, v, scale, ref)
    bad = err > tol
    worst = np.argmax(err - tol)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst err "
                           f"{err.flat[worst]:.3e} (tolerance {tol.flat[worst]:.3e}) at ref "
                           f"{ref.flat[worst]:.4f}")


def approx_magnitude(q_g, channels, kmin, kmax):
    """Per page: sum over the kept channels i of |q_g[i] * K_sel[i][page]|, where K_sel is the
    Kmax row when q_g[i] >= 0 and the Kmin row otherwise (the summary the score itself reads)."""
    q_g = np.asarray(q_g, dtype=np.float64)
    mag = np.zeros(kmin.shape[1], dtype=np.float64)
    for i in np.asarray(channels, dtype=np.int64):
        row = kmax[i] if q_g[i] >= 0 else kmin[i]
        mag += np.abs(q_g[i] * row)
    return mag


def fp32_gamma(n):
    """n u / (1 - n u) for fp32's unit roundoff u = 2^-24."""
    u = 2.0 ** -24
    return n * u / (1.0 - n * u)


def check_approx(gpu_scores, ref_scores, magnitude, n_channels, what="approx scores"):
    """magnitude: per page, sum over the kept channels of |q_g[i] * K_sel[i][page]|."""
    err = np.abs(np.asarray(gpu_scores, dtype=np.float64) - ref_scores)
    tol = 2.0 * fp32_gamma(n_channels + 9) * magnitude + 1e-30
    bad = err > tol
    worst = np.argmax(err - tol)
    assert not bad.any(), (f"{what}: {bad.sum()} outside tolerance; worst err "
                           f"{err.flat[worst]:.3e} (tolerance {tol.flat[worst]:.3e})")
