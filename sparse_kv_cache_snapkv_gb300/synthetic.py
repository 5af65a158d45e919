"""Seeded synthetic inputs for the RocketKV hot path (shared by tests, smoke and bench).

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic, so both the CUDA library and the CPU oracle can be fed from it.

Recipe (Llama-3.1-8B attention shapes: 32 query heads, 8 KV heads, head_dim 128, bf16):
  * K[t, c] = sigma[c] * z with sigma[c] ~ lognormal(0, 1) drawn per (sequence, layer, KV head,
    channel); V = z'. z, z' ~ N(0, 1). Optional outlier channels: `outliers` seeded channels per
    (unit, KV head) get sigma * 10.
  * u_g: a seeded unit vector per (unit, KV head), the mean direction of that group's window
    queries: Q_win[h, j] = z'' + u_g.
  * Needles: `needles` distinct seeded prefix positions per (unit, KV head) hold K = 4 ||sigma||_2
    u_g, a key aligned with the mean window-query direction.
  * Decode queries: plain N(0, 1). Appended decode tokens: K as above (same sigma), V ~ N(0, 1).
  * Positions past a sequence's length are zero.
  * A second conversation turn (`second_turn_inputs`): a new direction u2, window queries
    z'' + 4 u2, keys ||sigma||_2 u2 planted in the first prompt, and the turn's new input tokens.
A "unit" is one (sequence, layer) pair; units are sequence-major: u = s * layers + layer.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_seq: int
    n_layers: int
    n_kv: int
    gqa: int
    head_dim: int
    lens: tuple                 # per-sequence prompt length
    window: int
    budget: int
    page: int = 4
    channels: int = 32
    kernel: int = 0             # 0 = adaptive from each sequence's length
    decode_steps: int = 16
    append: bool = False
    needles: int = 8
    outliers: int = 0
    keep: int = 0               # 0 = planned: min(L, B * p * d / c)

    @property
    def n(self) -> int:
        return self.n_seq * self.n_layers

    @property
    def n_q(self) -> int:
        return self.n_kv * self.gqa

    @property
    def max_len(self) -> int:
        return max(self.lens)

    def with_layers(self, n_layers: int) -> "Workload":
        return replace(self, n_layers=n_layers)


def _ragged_lens(n: int, lo: int, hi: int, seed: int) -> tuple:
    g = torch.Generator().manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g).tolist())


WORKLOADS = {
    # batch 1, 8 q / 2 kv heads, 4K prompt, W 32, k 7, B 256, page 4, 32 of 128 channels.
    "tiny_4k": Workload("tiny_4k", 1, 1, 2, 4, 128, (4096,), 32, 256, kernel=7,
                        decode_steps=16, needles=8, keep=4096),
    # Llama-3.1-8B, all 32 layers, batch 1, 32K context, B 256, 128 decode steps.
    "llama8b_32k": Workload("llama8b_32k", 1, 32, 8, 4, 128, (32768,), 32, 256,
                            decode_steps=128, needles=64),
    # 128K context, batch 4, B 1024, 4 outlier channels per head at 10x.
    "llama8b_128k_b4": Workload("llama8b_128k_b4", 4, 32, 8, 4, 128, (131072,) * 4, 32, 1024,
                                decode_steps=64, needles=64, outliers=4),
    # 16 sequences of U[8K, 64K] tokens, 1 layer, B 512, 256 steps with appends.
    "ragged16": Workload("ragged16", 16, 1, 8, 4, 128, _ragged_lens(16, 8192, 65536, 4004), 32,
                         512, decode_steps=256, append=True, needles=64),
    # 128K prompt, W 64, 1 layer (kernel and budget swept by the caller).
    "prefill128k": Workload("prefill128k", 1, 1, 8, 4, 128, (131072,), 64, 1024, kernel=31,
                            decode_steps=0, needles=64),
}


def unit_lens(wl: Workload) -> List[int]:
    return [wl.lens[u // wl.n_layers] for u in range(wl.n)]


def prefill_inputs(wl: Workload, seed: int, device="cpu"):
    """K, V [n, Hkv, Lmax, d], Q_win [n, Hq, W, d] (bf16), seq_lens [n] int32, sigma, needles."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    n, hkv, d, lmax, W = wl.n, wl.n_kv, wl.head_dim, wl.max_len, wl.window
    lens = unit_lens(wl)
    f32 = dict(device=dev, dtype=torch.float32)
    sigma = torch.exp(torch.randn(n, hkv, d, generator=g, **f32))
    if wl.outliers:
        for u in range(n):
            for h in range(hkv):
                ch = torch.randperm(d, generator=g, device=dev)[: wl.outliers]
                sigma[u, h, ch] *= 10.0
    direction = torch.randn(n, hkv, d, generator=g, **f32)
    direction /= direction.norm(dim=-1, keepdim=True)
    k = torch.empty(n, hkv, lmax, d, device=dev, dtype=torch.bfloat16)
    v = torch.empty_like(k)
    needle_pos = torch.zeros(n, hkv, wl.needles, dtype=torch.int64)
    for u in range(n):
        L = lens[u]
        z = torch.randn(hkv, lmax, d, generator=g, **f32)
        z *= sigma[u][:, None, :]
        zv = torch.randn(hkv, lmax, d, generator=g, **f32)
        if L < lmax:
            z[:, L:] = 0
            zv[:, L:] = 0
        if wl.needles:
            for h in range(hkv):
                pos = torch.randperm(L - W, generator=g, device=dev)[: wl.needles]
                z[h, pos] = (4.0 * sigma[u, h].norm() * direction[u, h])[None, :]
                needle_pos[u, h] = pos.sort().values.cpu()
        k[u] = z.to(torch.bfloat16)
        v[u] = zv.to(torch.bfloat16)
        del z, zv
    qz = torch.randn(n, hkv, wl.gqa, W, d, generator=g, **f32)
    qz += direction[:, :, None, None, :]
    q_win = qz.reshape(n, hkv * wl.gqa, W, d).to(torch.bfloat16)
    seq_lens = torch.tensor(lens, dtype=torch.int32, device=dev)
    return {"k": k, "v": v, "q_win": q_win, "seq_lens": seq_lens, "sigma": sigma,
            "needles": needle_pos}


def second_turn_inputs(wl: Workload, x: dict, new_tokens: int, needles: int, seed: int,
                       device="cpu"):
    """Inputs of a second conversation turn, drawn after `prefill_inputs` (x):

    * u2: a new seeded unit vector per (unit, KV head); the turn's window queries are
      Q_win2[h, j] = z'' + 4 u2.
    * `needles` seeded positions of the first prompt's prefix (not its own needles) get
      K = ||sigma||_2 u2: keys of ordinary norm that only the second turn's queries single out.
      They are written into x["k"] in place, so draw the second turn before the first one runs.
    * new_k / new_v [n, Hkv, new_tokens, d] bf16: the turn's new input tokens, K = sigma * z,
      V = z' (the window queries belong to its last W tokens, so new_tokens >= W).
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    n, hkv, d, W = wl.n, wl.n_kv, wl.head_dim, wl.window
    assert new_tokens >= W
    lens = unit_lens(wl)
    f32 = dict(device=dev, dtype=torch.float32)
    sigma = x["sigma"].to(dev)
    direction = torch.randn(n, hkv, d, generator=g, **f32)
    direction /= direction.norm(dim=-1, keepdim=True)
    needle_pos = torch.zeros(n, hkv, needles, dtype=torch.int64)
    for u in range(n):
        L = lens[u]
        for h in range(hkv):
            taken = set(x["needles"][u, h].tolist())
            perm = torch.randperm(L - W, generator=g, device=dev).cpu().tolist()
            pos = sorted([p for p in perm if p not in taken][:needles])
            key = (sigma[u, h].norm() * direction[u, h]).to(torch.bfloat16)
            x["k"][u, h, pos] = key.to(x["k"].device)[None, :]
            needle_pos[u, h] = torch.tensor(pos, dtype=torch.int64)
    z = torch.randn(n, hkv, new_tokens, d, generator=g, **f32) * sigma[:, :, None, :]
    zv = torch.randn(n, hkv, new_tokens, d, generator=g, **f32)
    qz = torch.randn(n, hkv, wl.gqa, W, d, generator=g, **f32)
    qz += 4.0 * direction[:, :, None, None, :]
    return {"new_k": z.to(torch.bfloat16), "new_v": zv.to(torch.bfloat16),
            "q_win": qz.reshape(n, hkv * wl.gqa, W, d).to(torch.bfloat16), "needles": needle_pos}


def decode_queries(wl: Workload, steps: int, seed: int, device="cpu"):
    """[steps, n, Hq, d] bf16 decode queries, N(0, 1)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    return torch.randn(steps, wl.n, wl.n_q, wl.head_dim, generator=g, device=dev,
                       dtype=torch.float32).to(torch.bfloat16)


def append_tokens(wl: Workload, steps: int, sigma: torch.Tensor, seed: int, device="cpu"):
    """New decode K / V [steps, n, Hkv, d] bf16 (K scaled by the unit's sigma)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    shape = (steps, wl.n, wl.n_kv, wl.head_dim)
    nk = torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * sigma.to(dev)[None]
    nv = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    return nk.to(torch.bfloat16), nv.to(torch.bfloat16)


def random_cache(n: int, n_kv: int, cap: int, d: int, seed: int, device="cpu", scale_k=True):
    """A plain random compact cache [n, Hkv, cap, d] bf16 for decode-only tests."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    f32 = dict(device=dev, dtype=torch.float32)
    sigma = torch.exp(torch.randn(n, n_kv, 1, d, generator=g, **f32)) if scale_k else 1.0
    k = (torch.randn(n, n_kv, cap, d, generator=g, **f32) * sigma).to(torch.bfloat16)
    v = torch.randn(n, n_kv, cap, d, generator=g, **f32).to(torch.bfloat16)
    return k, v
