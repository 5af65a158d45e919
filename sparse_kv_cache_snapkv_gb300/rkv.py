"""Thin ctypes binding of librkv.so (include/rkv.h), one Python function per C entry point.

Argument marshalling only: shapes are read from the tensors, pointers and the current CUDA
stream are passed through, and any non-OK status raises RkvError. Every step of the hot path
runs in the library's kernels; there is no fallback of any kind. If the library is missing the
import fails with an explanation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

_lib = None

RKV_OK = 0
_STATUS = {0: "RKV_OK", 1: "RKV_ERR_INVALID_ARG", 2: "RKV_ERR_UNSUPPORTED",
           3: "RKV_ERR_WORKSPACE", 4: "RKV_ERR_CUDA", 5: "RKV_ERR_DEVICE_STATUS",
           6: "RKV_ERR_TOO_LARGE"}
STATUS_BYTES = 256
HEAD_DIM = 128

SYMBOLS = [
    "rkv_status_string", "rkv_check_status", "rkv_plan", "rkv_snapkv_workspace_bytes",
    "rkv_snapkv_compress", "rkv_summaries_workspace_bytes", "rkv_build_page_summaries",
    "rkv_hybrid_decode_workspace_bytes", "rkv_hybrid_decode",
    "rkv_dense_decode_workspace_bytes", "rkv_dense_decode", "rkv_dense_decode_noalloc",
    "rkv_build_page_summaries_mt", "rkv_hybrid_decode_mt", "rkv_plan_even_split",
    "rkv_snapkv_per_head_workspace_bytes", "rkv_snapkv_compress_per_head",
    "rkv_snapkv_compress_paged", "rkv_build_page_summaries_paged", "rkv_hybrid_decode_paged",
    "rkv_snapkv_compress_summarized", "rkv_snapkv_compress_avg_pool", "rkv_snapkv_select",
    "rkv_snapkv_scores", "rkv_testing_scores_wait_timeout", "rkv_testing_decode_layout",
]


class RkvError(RuntimeError):
    def __init__(self, fn: str, code: int, bits: int = 0):
        self.code = code
        self.bits = bits
        extra = f" (device bits 0x{bits:x})" if bits else ""
        super().__init__(f"{fn} -> {_STATUS.get(code, code)}{extra}")


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load librkv.so (optionally building it first)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError(f"librkv.so not found at {path}: run "
                              "`python -c 'import __graft_entry__ as g; g.build()'` first")
        _build.build()
    lib = ctypes.CDLL(path)
    vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    u32p = ctypes.POINTER(ctypes.c_uint32)
    ip = ctypes.POINTER(ctypes.c_int)
    sigs = {
        "rkv_status_string": ([i32], ctypes.c_char_p),
        "rkv_check_status": ([vp, vp, u32p], i32),
        "rkv_plan": ([i32, i32, i32, i32, i32, ip, ip, ip, ip], i32),
        "rkv_snapkv_workspace_bytes": ([i32, i32, i32, i32, i32], sz),
        "rkv_snapkv_compress": ([vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32,
                                 vp, vp, i32, vp, vp, vp, vp, sz, vp], i32),
        "rkv_snapkv_compress_avg_pool": ([vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                          i32, f32, vp, vp, i32, vp, vp, vp, vp, sz, vp], i32),
        "rkv_testing_scores_wait_timeout": ([vp, vp, vp, i32, i32, i32, i32, i32, i32, f32,
                                             vp, ctypes.c_uint64, vp, sz, vp], i32),
        "rkv_snapkv_scores": ([vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, vp, sz, vp],
                              i32),
        "rkv_testing_decode_layout": ([i32], i32),
        "rkv_snapkv_select": ([vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, vp, i32,
                               vp, vp, vp, sz, vp], i32),
        "rkv_summaries_workspace_bytes": ([], sz),
        "rkv_build_page_summaries": ([vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp,
                                      sz, vp], i32),
        "rkv_hybrid_decode_workspace_bytes": ([i32, i32, i32, i32, i32, i32], sz),
        "rkv_hybrid_decode": ([vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                               i32, i32, i32, f32, vp, vp, vp, vp, vp, sz, vp], i32),
        "rkv_dense_decode_workspace_bytes": ([i32, i32, i32, i32], sz),
        "rkv_dense_decode": ([vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, sz, vp],
                             i32),
        "rkv_dense_decode_noalloc": ([vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp],
                                     i32),
        "rkv_plan_even_split": ([i32, i32, i32, ip, ip, ip, ip], i32),
        "rkv_snapkv_per_head_workspace_bytes": ([i32, i32, i32, i32, i32], sz),
        "rkv_snapkv_compress_per_head": ([vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                          f32, vp, vp, i32, vp, vp, vp, vp, sz, vp], i32),
        "rkv_snapkv_compress_summarized": ([vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                            i32, f32, vp, vp, i32, vp, vp, vp, i32, i32, vp, vp,
                                            vp, sz, vp], i32),
        "rkv_snapkv_compress_paged": ([vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                       f32, vp, vp, i32, i32, vp, i32, vp, vp, vp, vp, sz, vp],
                                      i32),
        "rkv_build_page_summaries_paged": ([vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                            i32, vp, vp, vp, sz, vp], i32),
        "rkv_hybrid_decode_paged": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                     i32, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, sz,
                                     vp], i32),
        "rkv_build_page_summaries_mt": ([vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp,
                                         vp, vp, sz, vp], i32),
        "rkv_hybrid_decode_mt": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                  i32, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, sz, vp],
                                 i32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


# ------------------------------------------------------------------------------- helpers
def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("librkv takes device tensors only")
    if not t.is_contiguous():
        raise ValueError("librkv takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, code: int):
    if code != RKV_OK:
        raise RkvError(fn, code)


def _bf16(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")


def _group(hq: int, n_kv: int) -> int:
    """Query heads per KV head; the query heads must split evenly over the KV heads."""
    if n_kv <= 0 or hq % n_kv != 0:
        raise ValueError(f"{hq} query heads do not split over {n_kv} KV heads")
    return hq // n_kv


def workspace(nbytes: int, device) -> torch.Tensor:
    """A zeroed workspace (the device status word must start at zero)."""
    return torch.zeros(max(int(nbytes), STATUS_BYTES), dtype=torch.uint8, device=device)


def rkv_status_string(code: int) -> str:
    return load().rkv_status_string(code).decode()


def rkv_check_status(ws: torch.Tensor, stream=None) -> int:
    """Sync, read and clear the device status word; raise RkvError if it was non-zero."""
    bits = ctypes.c_uint32(0)
    code = load().rkv_check_status(_ptr(ws), _stream(stream), ctypes.byref(bits))
    if code != RKV_OK:
        raise RkvError("rkv_check_status", code, bits.value)
    return bits.value


def rkv_plan(ctx: int, budget: int, head_dim: int = HEAD_DIM, page: int = 0, channels: int = 0):
    """(keep, page, channels, kernel_size) for one sequence."""
    out = [ctypes.c_int(0) for _ in range(4)]
    code = load().rkv_plan(ctx, budget, head_dim, page, channels, *[ctypes.byref(o) for o in out])
    _check("rkv_plan", code)
    return tuple(o.value for o in out)


def rkv_plan_even_split(ctx: int, budget: int, head_dim: int = HEAD_DIM):
    """(keep, page, channels, kernel_size) from the even split of ctx / budget."""
    out = [ctypes.c_int(0) for _ in range(4)]
    code = load().rkv_plan_even_split(ctx, budget, head_dim, *[ctypes.byref(o) for o in out])
    _check("rkv_plan_even_split", code)
    return tuple(o.value for o in out)


# ------------------------------------------------------------------------------- stage 1
def rkv_snapkv_workspace_bytes(n: int, n_kv: int, gqa: int, max_len: int, window: int) -> int:
    return int(load().rkv_snapkv_workspace_bytes(n, n_kv, gqa, max_len, window))


def rkv_snapkv_compress(k, v, seq_lens, q_win, kernel_size: int, keep: int, scale: float,
                        k_out, v_out, kept_idx, out_len, scores_out=None, ws=None,
                        stream=None):
    """SnapKV++ compression of every (unit, KV head); see include/rkv.h."""
    _bf16(k, "k"), _bf16(v, "v"), _bf16(q_win, "q_win"), _i32(seq_lens, "seq_lens")
    _i32(kept_idx, "kept_idx"), _i32(out_len, "out_len")
    n, n_kv, max_len, d = k.shape
    hq, window = q_win.shape[1], q_win.shape[2]
    gqa = _group(hq, n_kv)
    cap = k_out.shape[2]
    if ws is None:
        ws = workspace(rkv_snapkv_workspace_bytes(n, n_kv, gqa, max_len, window), k.device)
    code = load().rkv_snapkv_compress(
        _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(q_win), n, n_kv, gqa, d, max_len, window,
        kernel_size, keep, float(scale), _ptr(k_out), _ptr(v_out), cap, _ptr(kept_idx),
        _ptr(out_len), _ptr(scores_out), _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_snapkv_compress", code)
    return ws


def rkv_snapkv_compress_avg_pool(k, v, seq_lens, q_win, kernel_size: int, keep: int,
                                 scale: float, k_out, v_out, kept_idx, out_len, scores_out=None,
                                 ws=None, stream=None):
    """SnapKV++ compression with average instead of max pooling; see include/rkv.h."""
    _bf16(k, "k"), _bf16(v, "v"), _bf16(q_win, "q_win"), _i32(seq_lens, "seq_lens")
    _i32(kept_idx, "kept_idx"), _i32(out_len, "out_len")
    n, n_kv, max_len, d = k.shape
    hq, window = q_win.shape[1], q_win.shape[2]
    gqa = _group(hq, n_kv)
    cap = k_out.shape[2]
    if ws is None:
        ws = workspace(rkv_snapkv_workspace_bytes(n, n_kv, gqa, max_len, window), k.device)
    code = load().rkv_snapkv_compress_avg_pool(
        _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(q_win), n, n_kv, gqa, d, max_len, window,
        kernel_size, keep, float(scale), _ptr(k_out), _ptr(v_out), cap, _ptr(kept_idx),
        _ptr(out_len), _ptr(scores_out), _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_snapkv_compress_avg_pool", code)
    return ws


def rkv_snapkv_select(k, seq_lens, q_win, kernel_size: int, keep: int, scale: float, kept_idx,
                      out_len, scores_out=None, ws=None, stream=None):
    """RocketKV-MT stage 1: scores, pooling and top-k over the full history, kept indices only
    (kept_idx [n][n_kv][kept_stride], kept_stride >= keep); see include/rkv.h."""
    _bf16(k, "k"), _bf16(q_win, "q_win"), _i32(seq_lens, "seq_lens")
    _i32(kept_idx, "kept_idx"), _i32(out_len, "out_len")
    n, n_kv, max_len, d = k.shape
    hq, window = q_win.shape[1], q_win.shape[2]
    gqa = _group(hq, n_kv)
    if ws is None:
        ws = workspace(rkv_snapkv_workspace_bytes(n, n_kv, gqa, max_len, window), k.device)
    code = load().rkv_snapkv_select(
        _ptr(k), _ptr(seq_lens), _ptr(q_win), n, n_kv, gqa, d, max_len, window, kernel_size,
        keep, float(scale), _ptr(kept_idx), kept_idx.shape[2], _ptr(out_len), _ptr(scores_out),
        _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_snapkv_select", code)
    return ws


def rkv_snapkv_scores(k, seq_lens, q_win, scale: float, scores_out, ws=None, stream=None):
    """Stage-1 window scores only (no pooling, selection or gather) into
    scores_out [n][n_kv][max_len - window] fp32; see include/rkv.h."""
    _bf16(k, "k"), _bf16(q_win, "q_win"), _i32(seq_lens, "seq_lens")
    n, n_kv, max_len, d = k.shape
    hq, window = q_win.shape[1], q_win.shape[2]
    gqa = _group(hq, n_kv)
    if ws is None:
        ws = workspace(rkv_snapkv_workspace_bytes(n, n_kv, gqa, max_len, window), k.device)
    code = load().rkv_snapkv_scores(
        _ptr(k), _ptr(seq_lens), _ptr(q_win), n, n_kv, gqa, d, max_len, window, float(scale),
        _ptr(scores_out), _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_snapkv_scores", code)
    return ws


def rkv_testing_scores_wait_timeout(k, seq_lens, q_win, scale: float, scores_out,
                                    wait_limit_ns: int, ws=None, stream=None):
    """Test hook (include/rkv_testing.h): the score passes with one K tile of block 0 never
    loaded, so that its bounded waits run out after wait_limit_ns."""
    _bf16(k, "k"), _bf16(q_win, "q_win"), _i32(seq_lens, "seq_lens")
    n, n_kv, max_len, d = k.shape
    hq, window = q_win.shape[1], q_win.shape[2]
    gqa = _group(hq, n_kv)
    if ws is None:
        ws = workspace(rkv_snapkv_workspace_bytes(n, n_kv, gqa, max_len, window), k.device)
    code = load().rkv_testing_scores_wait_timeout(
        _ptr(k), _ptr(seq_lens), _ptr(q_win), n, n_kv, gqa, d, max_len, window, float(scale),
        _ptr(scores_out), int(wait_limit_ns), _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_testing_scores_wait_timeout", code)
    return ws


def rkv_testing_decode_layout(layout: int) -> None:
    """Test hook (include/rkv_testing.h): the hybrid decode's shared-memory layout for later
    calls in this process (0 automatic, 1 ordinary, 2 wide wherever it fits)."""
    _check("rkv_testing_decode_layout", load().rkv_testing_decode_layout(int(layout)))


def rkv_snapkv_per_head_workspace_bytes(n: int, n_kv: int, gqa: int, max_len: int,
                                        window: int) -> int:
    return int(load().rkv_snapkv_per_head_workspace_bytes(n, n_kv, gqa, max_len, window))


def rkv_snapkv_compress_per_head(k, v, seq_lens, q_win, kernel_size: int, keep: int,
                                 scale: float, k_out, v_out, kept_idx, out_len, scores_out=None,
                                 ws=None, stream=None):
    """SnapKV without the GQA sum: every query head scored and filtered on its own; outputs per
    query head ([n][n_kv*gqa][...]); see include/rkv.h."""
    _bf16(k, "k"), _bf16(v, "v"), _bf16(q_win, "q_win"), _i32(seq_lens, "seq_lens")
    _i32(kept_idx, "kept_idx"), _i32(out_len, "out_len")
    n, n_kv, max_len, d = k.shape
    hq, window = q_win.shape[1], q_win.shape[2]
    gqa = _group(hq, n_kv)
    cap = k_out.shape[2]
    if ws is None:
        ws = workspace(rkv_snapkv_per_head_workspace_bytes(n, n_kv, gqa, max_len, window),
                       k.device)
    code = load().rkv_snapkv_compress_per_head(
        _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(q_win), n, n_kv, gqa, d, max_len, window,
        kernel_size, keep, float(scale), _ptr(k_out), _ptr(v_out), cap, _ptr(kept_idx),
        _ptr(out_len), _ptr(scores_out), _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_snapkv_compress_per_head", code)
    return ws


def rkv_snapkv_compress_summarized(k, v, seq_lens, q_win, kernel_size: int, keep: int,
                                   scale: float, k_out, v_out, kept_idx, out_len, page: int,
                                   kmin, kmax, scores_out=None, ws=None, stream=None):
    """rkv_snapkv_compress + page summaries of the compact cache in one pass."""
    _bf16(k, "k"), _bf16(v, "v"), _bf16(q_win, "q_win"), _i32(seq_lens, "seq_lens")
    _i32(kept_idx, "kept_idx"), _i32(out_len, "out_len"), _bf16(kmin, "kmin")
    n, n_kv, max_len, d = k.shape
    hq, window = q_win.shape[1], q_win.shape[2]
    gqa = _group(hq, n_kv)
    cap = k_out.shape[2]
    page_cap = kmin.shape[-1]
    if ws is None:
        ws = workspace(rkv_snapkv_workspace_bytes(n, n_kv, gqa, max_len, window), k.device)
    code = load().rkv_snapkv_compress_summarized(
        _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(q_win), n, n_kv, gqa, d, max_len, window,
        kernel_size, keep, float(scale), _ptr(k_out), _ptr(v_out), cap, _ptr(kept_idx),
        _ptr(out_len), _ptr(scores_out), page, page_cap, _ptr(kmin), _ptr(kmax), _ptr(ws),
        ws.numel(), _stream(stream))
    _check("rkv_snapkv_compress_summarized", code)
    return ws


# ------------------------------------------------------------------------------- stage 2
def rkv_build_page_summaries(k_cache, length, page: int, kmin, kmax, first_token: int = 0,
                             ws=None, stream=None):
    _bf16(k_cache, "k_cache"), _i32(length, "len")
    n, n_kv, cap, d = k_cache.shape
    page_cap = kmin.shape[-1]
    if ws is None:
        ws = workspace(STATUS_BYTES, k_cache.device)
    code = load().rkv_build_page_summaries(
        _ptr(k_cache), _ptr(length), n, n_kv, d, cap, page, page_cap, first_token, _ptr(kmin),
        _ptr(kmax), _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_build_page_summaries", code)
    return ws


def rkv_hybrid_decode_workspace_bytes(n, n_kv, gqa, page_cap, budget, page) -> int:
    return int(load().rkv_hybrid_decode_workspace_bytes(n, n_kv, gqa, page_cap, budget, page))


def rkv_hybrid_decode(q, k_cache, v_cache, length, kmin, kmax, budget: int, page: int,
                      channels: int, scale: float, out, new_k=None, new_v=None,
                      sel_channels=None, sel_pages=None, approx_scores=None, ws=None,
                      stream=None):
    """One hybrid sparse decode step (optionally appending new_k / new_v first)."""
    _bf16(q, "q"), _bf16(k_cache, "k_cache"), _i32(length, "len")
    n, n_kv, cap, d = k_cache.shape
    gqa = _group(q.shape[1], n_kv)
    page_cap = kmin.shape[-1]
    if ws is None:
        ws = workspace(rkv_hybrid_decode_workspace_bytes(n, n_kv, gqa, page_cap, budget, page),
                       q.device)
    code = load().rkv_hybrid_decode(
        _ptr(q), _ptr(new_k), _ptr(new_v), _ptr(k_cache), _ptr(v_cache), _ptr(length),
        _ptr(kmin), _ptr(kmax), n, n_kv, gqa, d, cap, page_cap, budget, page, channels,
        float(scale), _ptr(out), _ptr(sel_channels), _ptr(sel_pages), _ptr(approx_scores),
        _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_hybrid_decode", code)
    return ws


def rkv_build_page_summaries_mt(k_full, kept_idx, kept_len, page: int, kmin, kmax,
                                first_token: int = 0, ws=None, stream=None):
    """Page summaries of the kept sequence k_full[u][g][kept_idx[u][g][j]] (RocketKV-MT)."""
    _bf16(k_full, "k_full"), _i32(kept_idx, "kept_idx"), _i32(kept_len, "kept_len")
    n, n_kv, full_cap, d = k_full.shape
    kcap = kept_idx.shape[-1]
    page_cap = kmin.shape[-1]
    if ws is None:
        ws = workspace(STATUS_BYTES, k_full.device)
    code = load().rkv_build_page_summaries_mt(
        _ptr(k_full), _ptr(kept_idx), _ptr(kept_len), n, n_kv, d, full_cap, kcap, page, page_cap,
        first_token, _ptr(kmin), _ptr(kmax), _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_build_page_summaries_mt", code)
    return ws


def rkv_hybrid_decode_mt(q, k_full, v_full, full_len, kept_idx, kept_len, kmin, kmax,
                         budget: int, page: int, channels: int, scale: float, out, new_k=None,
                         new_v=None, sel_channels=None, sel_pages=None, approx_scores=None,
                         ws=None, stream=None):
    """One hybrid decode step over the kept sequence of the full cache (RocketKV-MT),
    optionally appending new_k / new_v to the full cache and the kept list first."""
    _bf16(q, "q"), _bf16(k_full, "k_full"), _i32(full_len, "full_len")
    _i32(kept_idx, "kept_idx"), _i32(kept_len, "kept_len")
    n, n_kv, full_cap, d = k_full.shape
    gqa = _group(q.shape[1], n_kv)
    kcap = kept_idx.shape[-1]
    page_cap = kmin.shape[-1]
    if ws is None:
        ws = workspace(rkv_hybrid_decode_workspace_bytes(n, n_kv, gqa, page_cap, budget, page),
                       q.device)
    code = load().rkv_hybrid_decode_mt(
        _ptr(q), _ptr(new_k), _ptr(new_v), _ptr(k_full), _ptr(v_full), _ptr(full_len),
        _ptr(kept_idx), _ptr(kept_len), _ptr(kmin), _ptr(kmax), n, n_kv, gqa, d, full_cap, kcap,
        page_cap, budget, page, channels, float(scale), _ptr(out), _ptr(sel_channels),
        _ptr(sel_pages), _ptr(approx_scores), _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_hybrid_decode_mt", code)
    return ws


# ------------------------------------------------------------------------------- paged cache
def rkv_snapkv_compress_paged(k, v, seq_lens, q_win, kernel_size: int, keep: int, scale: float,
                              k_pool, v_pool, block_table, kept_idx, out_len, scores_out=None,
                              ws=None, stream=None):
    """SnapKV++ compression whose kept rows go to the pools through the block table."""
    _bf16(k, "k"), _bf16(k_pool, "k_pool"), _i32(block_table, "block_table")
    _i32(kept_idx, "kept_idx"), _i32(out_len, "out_len"), _i32(seq_lens, "seq_lens")
    n, n_kv, max_len, d = k.shape
    hq, window = q_win.shape[1], q_win.shape[2]
    gqa = _group(hq, n_kv)
    num_blocks, _, block, _ = k_pool.shape
    max_blocks = block_table.shape[-1]
    if ws is None:
        ws = workspace(rkv_snapkv_workspace_bytes(n, n_kv, gqa, max_len, window), k.device)
    code = load().rkv_snapkv_compress_paged(
        _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(q_win), n, n_kv, gqa, d, max_len, window,
        kernel_size, keep, float(scale), _ptr(k_pool), _ptr(v_pool), num_blocks, block,
        _ptr(block_table), max_blocks, _ptr(kept_idx), _ptr(out_len), _ptr(scores_out), _ptr(ws),
        ws.numel(), _stream(stream))
    _check("rkv_snapkv_compress_paged", code)
    return ws


def rkv_build_page_summaries_paged(k_pool, block_table, length, page: int, kmin, kmax,
                                   first_token: int = 0, ws=None, stream=None):
    _bf16(k_pool, "k_pool"), _i32(block_table, "block_table"), _i32(length, "len")
    num_blocks, n_kv, block, d = k_pool.shape
    n, max_blocks = block_table.shape
    page_cap = kmin.shape[-1]
    if ws is None:
        ws = workspace(STATUS_BYTES, k_pool.device)
    code = load().rkv_build_page_summaries_paged(
        _ptr(k_pool), _ptr(block_table), _ptr(length), n, n_kv, d, num_blocks, block, max_blocks,
        page, page_cap, first_token, _ptr(kmin), _ptr(kmax), _ptr(ws), ws.numel(),
        _stream(stream))
    _check("rkv_build_page_summaries_paged", code)
    return ws


def rkv_hybrid_decode_paged(q, k_pool, v_pool, block_table, length, kmin, kmax, budget: int,
                            page: int, channels: int, scale: float, out, new_k=None, new_v=None,
                            sel_channels=None, sel_pages=None, approx_scores=None, ws=None,
                            stream=None):
    """One hybrid decode step over a paged cache (appending new_k / new_v first if given)."""
    _bf16(q, "q"), _bf16(k_pool, "k_pool"), _i32(block_table, "block_table"), _i32(length, "len")
    num_blocks, n_kv, block, d = k_pool.shape
    n, max_blocks = block_table.shape
    gqa = _group(q.shape[1], n_kv)
    page_cap = kmin.shape[-1]
    if ws is None:
        ws = workspace(rkv_hybrid_decode_workspace_bytes(n, n_kv, gqa, page_cap, budget, page),
                       q.device)
    code = load().rkv_hybrid_decode_paged(
        _ptr(q), _ptr(new_k), _ptr(new_v), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
        _ptr(length), _ptr(kmin), _ptr(kmax), n, n_kv, gqa, d, num_blocks, block, max_blocks,
        page_cap, budget, page, channels, float(scale), _ptr(out), _ptr(sel_channels),
        _ptr(sel_pages), _ptr(approx_scores), _ptr(ws), ws.numel(), _stream(stream))
    _check("rkv_hybrid_decode_paged", code)
    return ws


def rkv_dense_decode_workspace_bytes(n, n_kv, gqa, max_len) -> int:
    return int(load().rkv_dense_decode_workspace_bytes(n, n_kv, gqa, max_len))


def rkv_dense_decode(q, k, v, length, scale: float, out, ws=None, stream=None):
    """Full-KV decode attention over len[u] tokens."""
    _bf16(q, "q"), _bf16(k, "k"), _i32(length, "len")
    n, n_kv, max_len, d = k.shape
    gqa = _group(q.shape[1], n_kv)
    if ws is None:
        ws = workspace(rkv_dense_decode_workspace_bytes(n, n_kv, gqa, max_len), q.device)
    code = load().rkv_dense_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(length), n, n_kv, gqa, d,
                                   max_len, float(scale), _ptr(out), _ptr(ws), ws.numel(),
                                   _stream(stream))
    _check("rkv_dense_decode", code)
    return ws


def rkv_dense_decode_noalloc(q, k, v, length, scale: float, out, stream=None):
    """Dense decode without a workspace: the library's fixed device scratch holds the partials.
    For callers that cannot allocate; calls sharing the scratch must not overlap on the GPU."""
    _bf16(q, "q"), _bf16(k, "k"), _i32(length, "len")
    n, n_kv, max_len, d = k.shape
    gqa = _group(q.shape[1], n_kv)
    code = load().rkv_dense_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(length), n, n_kv, gqa,
                                           d, max_len, float(scale), _ptr(out), _stream(stream))
    _check("rkv_dense_decode_noalloc", code)
