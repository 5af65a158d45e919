"""The bounded-wait path of the kernels, made to run out without any GPU fault.

rkv_testing_scores_wait_timeout (include/rkv_testing.h) runs the stage-1 score passes with every
mbarrier wait bounded by a short limit and with one K tile of thread block 0 never requested. The
waits on that tile run out: the block records RKV_DEV_WAIT_TIMEOUT in the status word, lets its
issued copies land, frees its tensor memory and returns. The test checks that the host reads the
status bit, and that the context is still usable: a normal call afterwards returns RKV_OK with
scores that match the oracle.
"""
import math

import numpy as np
import pytest
import torch

from oracle import rocketkv as O

pytestmark = pytest.mark.gpu

D = 128
SCORE_REL = 1e-4


def test_score_wait_runs_out_and_context_survives():
    from sparse_kv_cache_snapkv_gb300 import rkv, synthetic as S
    rkv.load()
    lens = [4096, 3001]
    wl = S.Workload("t", 2, 1, 2, 4, D, tuple(lens), 32, 256, needles=2)
    x = S.prefill_inputs(wl, seed=990, device="cuda")
    n, n_kv, max_len, _ = x["k"].shape
    scale = 1.0 / math.sqrt(D)
    scores = torch.zeros(n, n_kv, max_len - 32, dtype=torch.float32, device="cuda")
    ws = rkv.rkv_testing_scores_wait_timeout(x["k"], x["seq_lens"], x["q_win"], scale, scores,
                                             wait_limit_ns=2_000_000)
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_check_status(ws)
    assert e.value.code == 5 and (e.value.bits & 0x4), e.value
    rkv.rkv_check_status(ws)  # the status word was cleared by the read

    # the same context, a normal call: no status bit, and the scores match the oracle
    scores2 = torch.full_like(scores, -1.0)
    ws2 = rkv.rkv_snapkv_scores(x["k"], x["seq_lens"], x["q_win"], scale, scores2)
    rkv.rkv_check_status(ws2)
    for u, L in enumerate(lens):
        for g in range(n_kv):
            k = x["k"][u, g, :L].double().cpu().numpy()
            q = x["q_win"][u, g * 4:(g + 1) * 4].double().cpu().numpy()
            ref = O.window_scores(k, q, scale)
            got = scores2[u, g, :L - 32].double().cpu().numpy()
            assert (np.abs(got - ref) <= SCORE_REL * np.abs(ref) + 1e-30).all(), (u, g)
