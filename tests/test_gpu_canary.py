"""Canary checks: every output of a compression + decode pass sits between guard units filled
with a known pattern, and the parts of each output that the contract leaves untouched (rows past
out_len, pages past the last summarised page, kept entries past keep) are pre-filled too. After
the calls every guard byte must be unchanged, so a write past a unit's end or past the documented
extent shows up here even when the values inside are right."""
import math

import pytest
import torch

pytestmark = pytest.mark.gpu

D = 128
CANARY_F = -12345.0


def _guarded(shape, dtype, fill):
    """A tensor of shape (n+2, ...) filled with `fill`; returns (whole, view of units 1..n)."""
    whole = torch.full((shape[0] + 2,) + tuple(shape[1:]), fill, dtype=dtype, device="cuda")
    return whole, whole[1:shape[0] + 1]


def _guards_intact(whole, fill, what):
    assert (whole[0] == fill).all(), f"{what}: leading guard unit written"
    assert (whole[-1] == fill).all(), f"{what}: trailing guard unit written"


@pytest.mark.parametrize("append", [False, True])
def test_outputs_stay_inside_their_extent(append):
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    rkv.load()
    steps = 3
    wl = S.Workload("canary", 3, 1, 2, 4, D, (5000, 700, 3333), 32, 256, needles=4)
    x = S.prefill_inputs(wl, seed=8100, device="cuda")
    n, n_kv, gqa, max_len = wl.n, wl.n_kv, wl.gqa, wl.max_len
    keep, page, channels, _ = rkv.rkv_plan(max_len, 256)
    cap = keep + (steps if append else 0) + 5  # spare rows that must stay untouched
    page_cap = ((cap + page - 1) // page + 7) // 8 * 8
    scale = 1.0 / math.sqrt(D)
    bf = torch.bfloat16
    kw, k_out = _guarded((n, n_kv, cap, D), bf, CANARY_F)
    vw, v_out = _guarded((n, n_kv, cap, D), bf, CANARY_F)
    keptw, kept = _guarded((n, n_kv, keep), torch.int32, -77)
    lenw, out_len = _guarded((n,), torch.int32, -77)
    minw, kmin = _guarded((n, n_kv, D, page_cap), bf, CANARY_F)
    maxw, kmax = _guarded((n, n_kv, D, page_cap), bf, CANARY_F)
    ws = rkv.rkv_snapkv_compress_summarized(x["k"], x["v"], x["seq_lens"], x["q_win"], 0, keep,
                                            scale, k_out, v_out, kept, out_len, page, kmin, kmax)
    rkv.rkv_check_status(ws)
    length = out_len.clone()
    S_pages = (256 // 2) // page
    outw, out = _guarded((n, n_kv * gqa, D), bf, CANARY_F)
    selw, sel_p = _guarded((n, n_kv, S_pages), torch.int32, -77)
    chw, sel_c = _guarded((n, n_kv, channels), torch.int32, -77)
    dq = S.decode_queries(wl, steps, seed=8101, device="cuda")
    nk = nv = None
    if append:
        nk, nv = S.append_tokens(wl, steps, x["sigma"], seed=8102, device="cuda")
    for t in range(steps):
        ws = rkv.rkv_hybrid_decode(dq[t], k_out, v_out, length, kmin, kmax, 256, page, channels,
                                   scale, out, new_k=nk[t] if append else None,
                                   new_v=nv[t] if append else None, sel_channels=sel_c,
                                   sel_pages=sel_p)
        rkv.rkv_check_status(ws)
    torch.cuda.synchronize()
    for whole, fill, what in ((kw, CANARY_F, "k_out"), (vw, CANARY_F, "v_out"),
                              (keptw, -77, "kept"), (lenw, -77, "out_len"),
                              (minw, CANARY_F, "kmin"), (maxw, CANARY_F, "kmax"),
                              (outw, CANARY_F, "out"), (selw, -77, "sel_pages"),
                              (chw, -77, "sel_channels")):
        _guards_intact(whole, fill, what)
    # untouched extents inside each unit
    final_len = length.cpu().tolist()
    for u in range(n):
        L = final_len[u]
        assert (k_out[u, :, L:] == CANARY_F).all(), f"unit {u}: k_out rows past the length"
        assert (v_out[u, :, L:] == CANARY_F).all(), f"unit {u}: v_out rows past the length"
        P = (L + page - 1) // page
        assert (kmin[u, :, :, P:] == CANARY_F).all(), f"unit {u}: kmin past the last page"
        assert (kmax[u, :, :, P:] == CANARY_F).all(), f"unit {u}: kmax past the last page"
    assert final_len == [min(L, keep) + (steps if append else 0) for L in (5000, 700, 3333)]
