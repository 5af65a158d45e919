"""One pass of the RocketKV hot path over a batch: SnapKV++ compression of every (unit, KV head),
page summaries of the compact cache, then `decode_steps` hybrid sparse decode steps (with a
decode-token append before each step when the workload appends).

Buffers are device tensors allocated here through torch (plumbing only); every step runs in
librkv's kernels through the C ABI.
"""
from __future__ import annotations

import math

import torch

from . import rkv
from .synthetic import Workload

D = 128


class HotPath:
    def __init__(self, wl: Workload, k, v, q_win, seq_lens, dec_q, new_k=None, new_v=None,
                 scale: float = 1.0 / math.sqrt(D), fuse_summaries: bool = True):
        rkv.load()
        self.fuse_summaries = fuse_summaries  # the gather builds the page summaries
        self.wl = wl
        self.k, self.v, self.q_win, self.seq_lens = k, v, q_win, seq_lens
        self.dec_q = dec_q            # [steps, n, Hq, d]
        self.new_k, self.new_v = new_k, new_v
        self.scale = scale
        dev = k.device
        n, n_kv = wl.n, wl.n_kv
        keep, page, channels, _ = rkv.rkv_plan(wl.max_len, wl.budget, D, wl.page, wl.channels)
        self.keep = wl.keep or keep
        self.page, self.channels = page, channels
        steps = dec_q.shape[0]
        self.cap = self.keep + (steps if wl.append else 0)
        self.page_cap = ((self.cap + page - 1) // page + 7) // 8 * 8
        self.k_out = torch.zeros(n, n_kv, self.cap, D, dtype=torch.bfloat16, device=dev)
        self.v_out = torch.zeros_like(self.k_out)
        self.kept = torch.empty(n, n_kv, self.keep, dtype=torch.int32, device=dev)
        self.out_len = torch.zeros(n, dtype=torch.int32, device=dev)
        self.length = torch.zeros(n, dtype=torch.int32, device=dev)   # decode-time length
        self.kmin = torch.zeros(n, n_kv, D, self.page_cap, dtype=torch.bfloat16, device=dev)
        self.kmax = torch.zeros_like(self.kmin)
        self.out = torch.empty(steps, n, wl.n_q, D, dtype=torch.bfloat16, device=dev)
        self.ws_snap = rkv.workspace(
            rkv.rkv_snapkv_workspace_bytes(n, n_kv, wl.gqa, wl.max_len, wl.window), dev)
        self.ws_sum = rkv.workspace(rkv.STATUS_BYTES, dev)
        self.ws_dec = rkv.workspace(rkv.rkv_hybrid_decode_workspace_bytes(
            n, n_kv, wl.gqa, self.page_cap, wl.budget, page), dev)

    # individual phases ------------------------------------------------------------------
    def compress(self):
        if self.fuse_summaries:
            rkv.rkv_snapkv_compress_summarized(self.k, self.v, self.seq_lens, self.q_win,
                                               self.wl.kernel, self.keep, self.scale, self.k_out,
                                               self.v_out, self.kept, self.out_len, self.page,
                                               self.kmin, self.kmax, ws=self.ws_snap)
        else:
            rkv.rkv_snapkv_compress(self.k, self.v, self.seq_lens, self.q_win, self.wl.kernel,
                                    self.keep, self.scale, self.k_out, self.v_out, self.kept,
                                    self.out_len, ws=self.ws_snap)

    def summaries(self):
        # The decode-time length starts at the stage-1 length. With appends it grows, so it
        # lives in its own array (a device-to-device copy); otherwise out_len is used as is.
        if self.wl.append:
            self.length.copy_(self.out_len)
        else:
            self.length = self.out_len
        if not self.fuse_summaries:
            rkv.rkv_build_page_summaries(self.k_out, self.length, self.page, self.kmin,
                                         self.kmax, ws=self.ws_sum)

    def rotate_decode_sets(self, sets: int):
        """Give the decode `sets` copies of the compact cache and its summaries; step t reads copy
        t % sets. All copies hold what the compression wrote (call after a compression; the
        compression rewrites copy 0 with the same values). With every layer batched into one
        launch, consecutive steps would otherwise re-read one small set of rows that stays in L2;
        in a model the other layers' work runs in between, so each step reads its rows from HBM.
        Only for workloads without appends (an appended token would reach one copy only)."""
        assert not self.wl.append, "decode sets are for workloads without appends"
        self.sets = [(self.k_out, self.v_out, self.kmin, self.kmax)]
        for _ in range(1, sets):
            self.sets.append(tuple(t.clone() for t in self.sets[0]))

    def decode(self, t: int):
        nk = self.new_k[t] if self.new_k is not None else None
        nv = self.new_v[t] if self.new_v is not None else None
        sets = getattr(self, "sets", None)
        k, v, kmin, kmax = (sets[t % len(sets)] if sets else
                            (self.k_out, self.v_out, self.kmin, self.kmax))
        rkv.rkv_hybrid_decode(self.dec_q[t], k, v, self.length, kmin, kmax, self.wl.budget,
                              self.page, self.channels, self.scale, self.out[t], new_k=nk,
                              new_v=nv, ws=self.ws_dec)

    def step(self):
        self.compress()
        self.summaries()
        for t in range(self.dec_q.shape[0]):
            self.decode(t)

    def check_status(self):
        for ws in (self.ws_snap, self.ws_sum, self.ws_dec):
            rkv.rkv_check_status(ws)

    # accounting ---------------------------------------------------------------------------
    def launches_per_step(self) -> int:
        """Kernel launches of one step: compression = score pass 1, LSE merge, score pass 2,
        select, gather (which also builds the page summaries unless fuse_summaries is off: then
        one summaries launch more); then one decode launch per step (an append is done inside
        the decode launch)."""
        return 5 + (0 if self.fuse_summaries else 1) + self.dec_q.shape[0]

    def decode_bytes_per_launch(self) -> int:
        """Algorithmic HBM bytes of one hybrid decode launch (all units), budget-implied:
        per (unit, KV head): c rows of ceil(N1/p) bf16 summary values (one of Kmin / Kmax per
        kept channel), (B/2) tokens of K and V rows, G query rows in and G output rows out."""
        wl = self.wl
        pages = (self.keep + self.page - 1) // self.page
        per = (self.channels * pages * 2 + (wl.budget // 2) * D * 2 * 2 + 2 * wl.gqa * D * 2)
        return wl.n * wl.n_kv * per

    def compress_bytes(self) -> int:
        """Algorithmic bytes of one compression: K read once, V rows of kept tokens read, kept
        K / V rows written, window queries read; with fused summaries also Kmin / Kmax written."""
        wl = self.wl
        units = wl.n * wl.n_kv
        summaries = 2 * D * (-(-self.keep // self.page)) * 2 if self.fuse_summaries else 0
        return (units * (wl.max_len * D * 2 + 3 * self.keep * D * 2 + summaries)
                + wl.n * wl.n_q * wl.window * D * 2)

    def compress_flops(self) -> int:
        """Tensor-core flops of the two score passes (2 GEMMs of (G*W) x L x d per unit)."""
        wl = self.wl
        return 2 * 2 * wl.n * wl.n_kv * wl.gqa * wl.window * wl.max_len * D
