"""Python binding of libzp, the Compressed PagedAttention hot path for GB300.

Argument marshalling only: every function forwards torch tensors' device
pointers and sizes to the C ABI declared in ``include/zp.h`` and raises
``ZPError`` on a non-OK status.  All arithmetic runs in the CUDA kernels of
libzp.so; there is no CPU fallback.  The library must have been built (see
``compressed_paged_kv_zp_gb300/_build.py`` or ``__graft_entry__.build()``):
importing this package without it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzp.so")

ZP_BF16 = 0
ZP_F32 = 1
_DTYPES = {torch.bfloat16: ZP_BF16, torch.float32: ZP_F32}

STATUS = {0: "ZP_OK", 1: "ZP_ERR_INVALID_ARG", 2: "ZP_ERR_SHAPE", 3: "ZP_ERR_DTYPE",
          4: "ZP_ERR_CAPACITY", 5: "ZP_ERR_CUDA", 6: "ZP_ERR_TIMEOUT", 7: "ZP_ERR_DEVICE"}

# every symbol include/*.h declares
EXPORTS = [
    "zp_last_error", "zp_status_string", "zp_version", "zp_device_status",
    "zp_decode_workspace_size", "zp_paged_decode_attn", "zp_paged_decode_attn_rho", "zp_paged_decode_attn_noalloc",
    "zp_debug_noalloc_preset_ctl", "zp_append_kv", "zp_needs_compression",
    "zp_needs_compression_batch",
    "zp_window_score_workspace_size", "zp_window_score",
    "zp_score_workspace_size", "zp_score_tokens", "zp_select_topk", "zp_compact_pages",
    "zp_compress_workspace_size", "zp_compress_layers", "zp_compress_layers_rho", "zp_compress_rho_supported",
    "zp_pool_create", "zp_pool_destroy", "zp_pool_num_free", "zp_pool_refcount", "zp_pool_alloc",
    "zp_pool_incref", "zp_pool_release", "zp_plan_compaction", "zp_plan_compaction_batch",
    "zp_plan_capacity",
    # include/zp_sched.h
    "zp_sched_create", "zp_sched_destroy", "zp_sched_add_request", "zp_sched_schedule", "zp_sched_commit",
    "zp_sched_take_compressions", "zp_sched_compression_done", "zp_sched_counts", "zp_sched_request_info",
]


class ZPError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), msg))
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("n_total_blocks", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class ScoreParams(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int32), ("use_global", ctypes.c_int32), ("alpha", ctypes.c_float),
                ("pool_kernel", ctypes.c_int32), ("pool_policy", ctypes.c_int32),
                ("use_similarity", ctypes.c_int32), ("lightning", ctypes.c_int32),
                ("threshold", ctypes.c_float), ("lambda_", ctypes.c_float), ("tau", ctypes.c_float)]


class ScoreRows(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("stride", ctypes.c_int64), ("layer_stride", ctypes.c_int64),
                ("rows", ctypes.c_void_p)]


class RhoRows(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("stride", ctypes.c_int64), ("layer_stride", ctypes.c_int64),
                ("rows", ctypes.c_void_p), ("n_rows", ctypes.c_int32), ("threshold", ctypes.c_float)]


def _rho_rows(rho, rows, threshold=0.0):
    """rho: float32 [R][h_kv][stride] or [layers][R][h_kv][stride]; rows: int32 device or None."""
    if rho.dtype != torch.float32 or rho.dim() not in (3, 4):
        raise ValueError("redundancy rows must be float32 [R][h_kv][stride] or [layers][R][h_kv][stride]")
    if rows is not None and rows.dtype != torch.int32:
        raise ValueError("rho_rows must be int32")
    layer_stride = rho.stride(0) if rho.dim() == 4 else 0
    return ctypes.byref(RhoRows(_dev(rho, "rho").value, int(rho.shape[-1]), int(layer_stride),
                                _dev(rows, "rho_rows").value if rows is not None else None,
                                int(rho.shape[-3]), float(threshold)))


def _score_rows(attn, rows):
    """attn: float32 [R][h_kv][stride] or [layers][R][h_kv][stride]; rows: int32 [n] or None."""
    if attn is None:
        return None
    if attn.dtype != torch.float32 or attn.dim() not in (3, 4):
        raise ValueError("score rows must be float32 [R][h_kv][stride] or [layers][R][h_kv][stride]")
    if rows is not None and rows.dtype != torch.int32:
        raise ValueError("rows must be int32")
    layer_stride = attn.stride(0) if attn.dim() == 4 else 0
    return ctypes.byref(ScoreRows(_dev(attn, "attn").value, int(attn.shape[-1]), int(layer_stride),
                                  _dev(rows, "rows").value if rows is not None else None))


def score_params(window=16, use_global=True, alpha=0.8, pool_kernel=7, pool_policy=1,
                 use_similarity=True, lightning=True, threshold=0.9, lam=0.2, tau=0.4) -> ScoreParams:
    return ScoreParams(int(window), int(bool(use_global)), float(alpha), int(pool_kernel),
                       int(pool_policy), int(bool(use_similarity)), int(bool(lightning)),
                       float(threshold), float(lam), float(tau))


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("libzp.so is not built (expected at %s); run "
                          "compressed_paged_kv_zp_gb300._build.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(CacheDesc)
    lib.zp_last_error.restype = ctypes.c_char_p
    lib.zp_status_string.restype = ctypes.c_char_p
    lib.zp_status_string.argtypes = [ctypes.c_int]
    lib.zp_device_status.argtypes = [P, P, I32]
    lib.zp_decode_workspace_size.restype = SZ
    lib.zp_decode_workspace_size.argtypes = [D, I32, I32]
    lib.zp_paged_decode_attn.argtypes = [D, P, P, P, P, I32, P, I32, P, P, P, I32, I32, P, SZ, P]
    lib.zp_paged_decode_attn_rho.argtypes = [D, P, P, P, P, I32, P, I32, P, P, P, I32, I32, P, P, SZ, P]
    lib.zp_paged_decode_attn_noalloc.argtypes = [D, P, P, P, P, I32, P, I32, P, P, P, I32, I32, P]
    lib.zp_debug_noalloc_preset_ctl.argtypes = [I32, ctypes.c_uint64]
    lib.zp_append_kv.argtypes = [D, P, P, P, P, P, I32, P, I32, P]
    lib.zp_needs_compression.argtypes = [I32, I32, I32]
    lib.zp_needs_compression_batch.argtypes = [P, P, I32, I32, I32, P, P, P]
    lib.zp_score_workspace_size.restype = SZ
    lib.zp_score_workspace_size.argtypes = [D, I32, I32]
    lib.zp_window_score_workspace_size.restype = SZ
    lib.zp_window_score_workspace_size.argtypes = [D, I32, I32, I32]
    lib.zp_window_score.argtypes = [D, P, I32, P, P, I32, P, I32, P, I32, P, SZ, P]
    lib.zp_score_tokens.argtypes = [D, ctypes.POINTER(ScoreParams), P, P, I32, P, P, I32, P, P, P,
                                    I32, P, SZ, P]
    lib.zp_select_topk.argtypes = [P, I32, I32, P, I32, I32, P, P, P, P]
    lib.zp_compact_pages.argtypes = [D, P, P, I64, I32, P, I64, P, P, I32, P, I32, P, P, I32, P, I32, P]
    lib.zp_compress_workspace_size.restype = SZ
    lib.zp_compress_workspace_size.argtypes = [D, I32, I32, I32]
    lib.zp_compress_layers.argtypes = [D, ctypes.POINTER(ScoreParams), P, P, I64, I32, P, I32, P, P, I32, P, P,
                                       I64, P, I32, I32, P, P, P, P, I32, P, SZ, P]
    lib.zp_compress_rho_supported.restype = I32
    lib.zp_compress_rho_supported.argtypes = [D, ctypes.POINTER(ScoreParams), I32, I32]
    lib.zp_compress_layers_rho.argtypes = [D, ctypes.POINTER(ScoreParams), P, P, I64, I32, P, I32, P, P, I32, P,
                                           P, I64, P, I32, I32, P, P, P, P, I32, P, P]
    lib.zp_pool_create.restype = P
    lib.zp_pool_create.argtypes = [I32]
    lib.zp_pool_destroy.argtypes = [P]
    lib.zp_pool_num_free.argtypes = [P]
    lib.zp_pool_refcount.argtypes = [P, I32]
    lib.zp_pool_alloc.argtypes = [P, I32, P]
    lib.zp_pool_incref.argtypes = [P, I32, P]
    lib.zp_pool_release.argtypes = [P, I32, P]
    lib.zp_plan_compaction.argtypes = [P, P, I32, I32, P, P, P, P, P]
    lib.zp_plan_compaction_batch.argtypes = [P, P, I32, P, I32, I32, P, P, P, P, P, P]
    lib.zp_plan_capacity.argtypes = [I64, I64, I64, I32, I64, I64, P, P]
    return lib


lib = _load()


def _check(status: int) -> None:
    if status != 0:
        raise ZPError(status, lib.zp_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libzp must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t: Optional[torch.Tensor], name: str):
    if t is not None and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    return _ptr(t)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def cache_desc(h_q, h_kv, head_dim, block_size, n_total_blocks, dtype) -> CacheDesc:
    code = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return CacheDesc(int(h_q), int(h_kv), int(head_dim), int(block_size), int(n_total_blocks), code)


# ----------------------------------------------------------------------------- decode
def zp_decode_workspace_size(desc: CacheDesc, B: int, table_stride: int) -> int:
    n = lib.zp_decode_workspace_size(ctypes.byref(desc), int(B), int(table_stride))
    if n == 0 and B > 0:
        raise ZPError(2, lib.zp_last_error().decode() or "unsupported decode shape")
    return int(n)


def _slot_map(score_accum, score_rows):
    """(pointer, row count) of an optional int32 [B] slot map into score_accum [R][h_kv][stride]."""
    if score_rows is None:
        return None, 0
    if score_rows.dtype != torch.int32:
        raise ValueError("score_rows must be int32")
    if score_accum is None:
        raise ValueError("score_rows needs score_accum")
    return _dev(score_rows, "score_rows"), int(score_accum.shape[0])


def zp_paged_decode_attn(desc, q, k_cache, v_cache, block_table, seq_lens, out, score_accum=None,
                         window=0, workspace=None, stream=None, score_rows=None, rho=None, rho_rows=None,
                         rho_threshold=0.9) -> None:
    """score_rows: optional int32 [B] device map of batch entries to rows of
    score_accum (query slots); -1 = no slot, the entry is not scored.
    rho (optional float32 [R][h_kv][stride]) with rho_rows (int32 [B] device,
    -1 = none): the lightning redundancy row sums of the entries that have a
    row, at threshold rho_threshold (zp_paged_decode_attn_rho)."""
    B, table_stride = int(block_table.shape[0]), int(block_table.shape[1])
    rows_p, n_rows = _slot_map(score_accum, score_rows)
    if workspace is None:
        workspace = torch.empty(zp_decode_workspace_size(desc, B, table_stride), dtype=torch.uint8,
                                device=q.device)
    args = (ctypes.byref(desc), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_table, "block_table"), table_stride, _dev(seq_lens, "seq_lens"), B, _dev(out, "out"),
            _dev(score_accum, "score_accum"), rows_p, n_rows, int(window))
    tail = (_dev(workspace, "workspace"), workspace.numel(), _stream(stream))
    if rho is None:
        _check(lib.zp_paged_decode_attn(*args, *tail))
    else:
        if rho_rows is None or rho_rows.numel() != B:
            raise ValueError("rho needs rho_rows: one int32 entry per batch entry")
        _check(lib.zp_paged_decode_attn_rho(*args, _rho_rows(rho, rho_rows, rho_threshold), *tail))


def zp_paged_decode_attn_noalloc(desc, q, k_cache, v_cache, block_table, seq_lens, out,
                                 score_accum=None, window=0, stream=None, score_rows=None) -> None:
    """zp_paged_decode_attn with the library's built-in scratch (no workspace)."""
    B, table_stride = int(block_table.shape[0]), int(block_table.shape[1])
    rows_p, n_rows = _slot_map(score_accum, score_rows)
    _check(lib.zp_paged_decode_attn_noalloc(ctypes.byref(desc), _dev(q, "q"), _dev(k_cache, "k_cache"),
                                            _dev(v_cache, "v_cache"), _dev(block_table, "block_table"),
                                            table_stride, _dev(seq_lens, "seq_lens"), B, _dev(out, "out"),
                                            _dev(score_accum, "score_accum"), rows_p, n_rows, int(window),
                                            _stream(stream)))


def zp_append_kv(desc, k_new, v_new, k_cache, v_cache, block_table, seq_lens, stream=None) -> None:
    B, table_stride = int(block_table.shape[0]), int(block_table.shape[1])
    _check(lib.zp_append_kv(ctypes.byref(desc), _dev(k_new, "k_new"), _dev(v_new, "v_new"),
                            _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                            _dev(block_table, "block_table"), table_stride, _dev(seq_lens, "seq_lens"),
                            B, _stream(stream)))


# ----------------------------------------------------------------------------- compression
def zp_needs_compression(seq_len: int, block_size: int, max_blocks: int) -> bool:
    return bool(lib.zp_needs_compression(int(seq_len), int(block_size), int(max_blocks)))


def zp_needs_compression_batch(seq_lens, block_size: int, max_blocks: int, active=None,
                               max_blocks_seq=None):
    """Indices (int64 numpy array, ascending) of the sequences whose trigger
    holds; host numpy arrays in, no device work."""
    import numpy as np
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    n = int(lens.shape[0])
    act = None if active is None else np.ascontiguousarray(active, dtype=np.uint8)
    per = None if max_blocks_seq is None else np.ascontiguousarray(max_blocks_seq, dtype=np.int32)
    out = np.empty(max(n, 1), dtype=np.int32)
    cnt = ctypes.c_int32(0)
    _check(lib.zp_needs_compression_batch(lens.ctypes.data, None if act is None else act.ctypes.data, n,
                                          int(block_size), int(max_blocks),
                                          None if per is None else per.ctypes.data, out.ctypes.data,
                                          ctypes.byref(cnt)))
    return out[:cnt.value].astype(np.int64)


def zp_score_workspace_size(desc: CacheDesc, n: int, Lmax: int) -> int:
    return int(lib.zp_score_workspace_size(ctypes.byref(desc), int(n), int(Lmax)))


def zp_window_score_workspace_size(desc: CacheDesc, n: int, Lmax: int, window: int) -> int:
    return int(lib.zp_window_score_workspace_size(ctypes.byref(desc), int(n), int(Lmax), int(window)))


def zp_window_score(desc, q_window, k_cache, block_table, seq_lens, scores_out, workspace=None,
                    stream=None) -> None:
    n, table_stride = int(block_table.shape[0]), int(block_table.shape[1])
    window = int(q_window.shape[1])
    Lmax = int(scores_out.shape[-1])
    if workspace is None:
        workspace = torch.empty(max(zp_window_score_workspace_size(desc, n, Lmax, window), 1),
                                dtype=torch.uint8, device=scores_out.device)
    _check(lib.zp_window_score(ctypes.byref(desc), _dev(q_window, "q_window"), window,
                               _dev(k_cache, "k_cache"), _dev(block_table, "block_table"), table_stride,
                               _dev(seq_lens, "seq_lens"), n, _dev(scores_out, "scores_out"), Lmax,
                               _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))


def zp_score_tokens(desc, params: ScoreParams, k_cache, block_table, seq_lens, first_compression,
                    attn, global_F, scores_out, rows=None, workspace=None, stream=None) -> None:
    """attn: the attention-score rows, float32 [R][h_kv][stride] (the decode
    score_accum, or the output of zp_window_score); sequence i reads row
    rows[i] (rows None: row i).  On return the rows hold the global score."""
    n, table_stride = int(block_table.shape[0]), int(block_table.shape[1])
    Lmax = int(scores_out.shape[-1])
    if workspace is None:
        workspace = torch.empty(max(zp_score_workspace_size(desc, n, Lmax), 1), dtype=torch.uint8,
                                device=scores_out.device)
    if attn is None:
        raise ValueError("attn (the attention-score rows) is required")
    _check(lib.zp_score_tokens(ctypes.byref(desc), ctypes.byref(params), _dev(k_cache, "k_cache"),
                               _dev(block_table, "block_table"), table_stride,
                               _dev(seq_lens, "seq_lens"), _dev(first_compression, "first_compression"),
                               n, _score_rows(attn, rows), _dev(global_F, "global_F"),
                               _dev(scores_out, "scores_out"), Lmax, _dev(workspace, "workspace"),
                               workspace.numel(), _stream(stream)))


def zp_select_topk(scores, seq_lens, k, keep_idx, tie_count=None, k_seq=None, stream=None) -> None:
    """k_seq: optional int32 [n] device array of per-request budgets k_i <= k;
    keep_idx rows keep stride k and are padded with -1 after k_i."""
    n, h_kv, Lmax = (int(x) for x in scores.shape)
    _check(lib.zp_select_topk(_dev(scores, "scores"), h_kv, Lmax, _dev(seq_lens, "seq_lens"), n,
                              int(k), _dev(k_seq, "k_seq"), _dev(keep_idx, "keep_idx"),
                              _dev(tie_count, "tie_count"), _stream(stream)))


def zp_compact_pages(desc, k_base, v_base, layer_stride, layer_count, global_F, F_layer_stride,
                     src_table, dst_targets, seq_lens, keep_idx, k, scores=None, rows=None,
                     k_seq=None, stream=None) -> None:
    """scores/rows: the score rows zp_score_tokens left (float32 [R][h_kv][stride],
    or [layers][R][h_kv][stride] for several layers); needed when global_F is set."""
    n, table_stride = int(src_table.shape[0]), int(src_table.shape[1])
    _check(lib.zp_compact_pages(ctypes.byref(desc), _dev(k_base, "k_base"), _dev(v_base, "v_base"),
                                int(layer_stride), int(layer_count), _dev(global_F, "global_F"),
                                int(F_layer_stride), _score_rows(scores, rows),
                                _dev(src_table, "src_table"), table_stride,
                                _dev(dst_targets, "dst_targets"), int(dst_targets.shape[1]),
                                _dev(seq_lens, "seq_lens"), _dev(keep_idx, "keep_idx"), int(k),
                                _dev(k_seq, "k_seq"), n, _stream(stream)))


def zp_compress_workspace_size(desc: CacheDesc, n: int, Lmax: int, layer_count: int = 1) -> int:
    return int(lib.zp_compress_workspace_size(ctypes.byref(desc), int(n), int(Lmax), int(layer_count)))


def zp_compress_layers(desc, params: ScoreParams, k_cache, v_cache, block_table, seq_lens, first_compression,
                       attn, global_F, dst_targets, k, keep_idx, Lmax, rows=None, tie_count=None, scores_out=None,
                       workspace=None, k_seq=None, stream=None, rho=None, rho_rows=None) -> None:
    """Scores, keep sets and moves of one or several layers in one call.
    k_cache/v_cache: one layer [N_total][b][h_kv][d] or several
    [layers][N_total][b][h_kv][d]; global_F and attn (score rows) alike;
    keep_idx int32 [layers][n][h_kv][k] (or [n][h_kv][k] for one layer);
    k_seq: optional int32 [n] device array of per-request budgets k_i <= k.
    rho (optional float32 [R][h_kv][stride], or [layers][R][h_kv][stride]) with
    rho_rows (int32 [n] device or None: row i): lightning row sums written by
    the decode; the call then runs zp_compress_layers_rho (no workspace)."""
    n, table_stride = int(block_table.shape[0]), int(block_table.shape[1])
    layers = int(k_cache.shape[0]) if k_cache.dim() == 5 else 1
    layer_stride = int(k_cache.stride(0)) if layers > 1 else 0
    F_layer = int(global_F.stride(0)) if (global_F is not None and global_F.dim() == 4) else 0
    if layers > 1 and attn.dim() != 4:
        raise ValueError("several layers need score rows [layers][R][h_kv][stride]")
    if rho is not None:
        if layers > 1 and rho.dim() != 4:
            raise ValueError("several layers need redundancy rows [layers][R][h_kv][stride]")
        _check(lib.zp_compress_layers_rho(ctypes.byref(desc), ctypes.byref(params), _dev(k_cache, "k_cache"),
                                          _dev(v_cache, "v_cache"), layer_stride, layers,
                                          _dev(block_table, "block_table"), table_stride, _dev(seq_lens, "seq_lens"),
                                          _dev(first_compression, "first_compression"), n, _score_rows(attn, rows),
                                          _dev(global_F, "global_F"), F_layer, _dev(dst_targets, "dst_targets"),
                                          int(dst_targets.shape[1]), int(k), _dev(k_seq, "k_seq"),
                                          _dev(keep_idx, "keep_idx"), _dev(tie_count, "tie_count"),
                                          _dev(scores_out, "scores_out"), int(Lmax), _rho_rows(rho, rho_rows),
                                          _stream(stream)))
        return
    if workspace is None:
        workspace = torch.empty(max(zp_compress_workspace_size(desc, n, Lmax, layers), 1), dtype=torch.uint8,
                                device=k_cache.device)
    _check(lib.zp_compress_layers(ctypes.byref(desc), ctypes.byref(params), _dev(k_cache, "k_cache"),
                                  _dev(v_cache, "v_cache"), layer_stride, layers, _dev(block_table, "block_table"),
                                  table_stride, _dev(seq_lens, "seq_lens"),
                                  _dev(first_compression, "first_compression"), n, _score_rows(attn, rows),
                                  _dev(global_F, "global_F"), F_layer, _dev(dst_targets, "dst_targets"),
                                  int(dst_targets.shape[1]), int(k), _dev(k_seq, "k_seq"),
                                  _dev(keep_idx, "keep_idx"),
                                  _dev(tie_count, "tie_count"), _dev(scores_out, "scores_out"), int(Lmax),
                                  _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))


def zp_compress_rho_supported(desc, params: ScoreParams, Lmax: int, k: int) -> bool:
    """Whether zp_compress_layers_rho (the decode's row sums, one kernel) covers
    this cache, these switches, Lmax and k on the current device."""
    return bool(lib.zp_compress_rho_supported(ctypes.byref(desc), ctypes.byref(params), int(Lmax), int(k)))


def zp_plan_capacity(m_available: int, m_kv_block: int, m_q_request: int, max_blocks: int,
                     extra=(0, 1)):
    """(M, N_total) of eq. (1) / (2): the largest request concurrency and the
    block count for a memory budget; extra = (num, den) per-block overhead of
    the global score cache relative to K and V."""
    M, N = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib.zp_plan_capacity(int(m_available), int(m_kv_block), int(m_q_request), int(max_blocks),
                                int(extra[0]), int(extra[1]), ctypes.byref(M), ctypes.byref(N)))
    return M.value, N.value


def zp_device_status(clear: bool = True):
    code, detail = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib.zp_device_status(ctypes.byref(code), ctypes.byref(detail), int(bool(clear))))
    return code.value, detail.value


# ----------------------------------------------------------------------------- host pool
def _i32buf(n):
    return (ctypes.c_int32 * max(int(n), 1))()


class Pool:
    """Host block pool (zp_pool_*): reference counts and the free list."""

    def __init__(self, n_total: int):
        self._p = lib.zp_pool_create(int(n_total))
        if not self._p:
            raise ZPError(1, lib.zp_last_error().decode())
        self.n_total = int(n_total)

    def __del__(self):
        p = getattr(self, "_p", None)
        if p:
            lib.zp_pool_destroy(p)
            self._p = None

    @property
    def num_free(self) -> int:
        return int(lib.zp_pool_num_free(self._p))

    def refcount(self, block: int) -> int:
        return int(lib.zp_pool_refcount(self._p, int(block)))

    def alloc(self, n: int):
        buf = _i32buf(n)
        _check(lib.zp_pool_alloc(self._p, int(n), buf))
        return list(buf)[: int(n)]

    def incref(self, ids):
        ids = list(ids)
        buf = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(lib.zp_pool_incref(self._p, len(ids), buf))

    def release(self, ids):
        ids = list(ids)
        buf = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(lib.zp_pool_release(self._p, len(ids), buf))

    def plan_compaction(self, table, max_blocks: int):
        table = [int(x) for x in table]
        tb = (ctypes.c_int32 * max(len(table), 1))(*table)
        targets, new_table = _i32buf(max_blocks - 1), _i32buf(max_blocks)
        dropped = _i32buf(len(table))
        nd, nf = ctypes.c_int32(0), ctypes.c_int32(0)
        _check(lib.zp_plan_compaction(self._p, tb, len(table), int(max_blocks), targets, new_table,
                                      dropped, ctypes.byref(nd), ctypes.byref(nf)))
        return {"targets": list(targets)[: max_blocks - 1], "new_table": list(new_table)[:max_blocks],
                "dropped": list(dropped)[: nd.value], "n_fresh": nf.value}

    def plan_compaction_batch(self, tables, n_blocks, max_blocks: int, out=None, max_blocks_seq=None):
        """Plans of n sequences in one C call; tables int32 [n][stride] and
        n_blocks int32 [n] as numpy arrays; max_blocks_seq: optional int32 [n]
        per-request block budgets in [2, max_blocks] (rows padded with -1).
        Returns numpy arrays (reused from ``out`` when given): targets
        [n][max_blocks-1], new_tables [n][max_blocks], dropped [n][stride],
        n_dropped [n], n_fresh [n]."""
        import numpy as np
        tables = np.ascontiguousarray(tables, dtype=np.int32)
        n_blocks = np.ascontiguousarray(n_blocks, dtype=np.int32)
        n, stride = tables.shape
        if out is None:
            out = {"targets": np.empty((n, max_blocks - 1), np.int32),
                   "new_tables": np.empty((n, max_blocks), np.int32),
                   "dropped": np.empty((n, stride), np.int32), "n_dropped": np.empty(n, np.int32),
                   "n_fresh": np.empty(n, np.int32)}
        P = lambda a: ctypes.c_void_p(a.ctypes.data)  # noqa: E731
        mbs = None
        if max_blocks_seq is not None:
            mbs = np.ascontiguousarray(max_blocks_seq, dtype=np.int32)
            if mbs.shape != (n,):
                raise ValueError("max_blocks_seq must have one entry per sequence")
        _check(lib.zp_plan_compaction_batch(self._p, P(tables), stride, P(n_blocks), n, int(max_blocks),
                                            None if mbs is None else P(mbs), P(out["targets"]), P(out["new_tables"]), P(out["dropped"]),
                                            P(out["n_dropped"]), P(out["n_fresh"])))
        return out


__all__ = ["lib", "LIB_PATH", "EXPORTS", "ZPError", "CacheDesc", "ScoreParams", "ScoreRows", "RhoRows", "score_params",
           "cache_desc", "zp_decode_workspace_size", "zp_paged_decode_attn",
           "zp_paged_decode_attn_noalloc", "zp_append_kv",
           "zp_needs_compression", "zp_needs_compression_batch", "zp_window_score_workspace_size", "zp_window_score",
           "zp_score_workspace_size", "zp_score_tokens", "zp_select_topk",
           "zp_compact_pages", "zp_compress_workspace_size", "zp_compress_layers", "zp_compress_rho_supported", "zp_plan_capacity", "zp_device_status", "Pool",
           "ZP_BF16", "ZP_F32"]
