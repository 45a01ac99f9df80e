"""CPU oracle for the Compressed PagedAttention hot path (test infrastructure).

The arithmetic lives in ``zp_oracle.c`` (plain loops, fp64).  This module only
builds that file with gcc, loads it with ctypes and marshals numpy arrays; the
composition of the scoring steps in the paper's order is in ``pipeline.py``.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and this
package never imports the product.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zp_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_int = ctypes.c_int
_dbl = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile zp_oracle.c into liboracle.so next to it (gcc, no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.orc_decode_attention.argtypes = [_int, _int, _int, _int, _int, _f32p, _f32p, _f32p,
                                                 _i32p, _int, _i32p, _f64p, _f64p, _int]
            lib.orc_accumulate_window_score.argtypes = [_int, _int, _int, _int, _int, _i32p, _int,
                                                        _i32p, _f64p, _int, _f64p]
            lib.orc_window_score.argtypes = [_int, _int, _int, _int, _int, _f32p, _f32p, _i32p,
                                             _int, _f64p]
            lib.orc_global_score.argtypes = [_int, _int, _int, _int, _dbl, _i32p, _f64p, _f64p]
            lib.orc_max_pool.argtypes = [_int, _int, _f64p, _f64p]
            lib.orc_redundancy.argtypes = [_int, _int, _int, _f32p, _dbl, _dbl, _int, _f64p]
            lib.orc_redundancy_rho.argtypes = [_int, _int, _int, _f32p, _dbl, _int, _f64p]
            lib.orc_redundancy_rho_rows.argtypes = [_int, _int, _f32p, _dbl, _i32p, _int, _f64p]
            lib.orc_combine_and_window.argtypes = [_int, _int, _dbl, _f64p, _f64p]
            lib.orc_topk_keep.argtypes = [_int, _int, _f64p, _i32p, _u8p]
            lib.orc_compact_alg4.argtypes = [_u8p, ctypes.c_size_t, _int, _int, _int, _i32p, _int,
                                             _i32p, _u8p]
            lib.orc_needs_compression.argtypes = [_int, _int, _int]
            lib.orc_plan_targets.argtypes = [_i32p, _int, _int, _i32p, _i32p, _int, _i32p, _i32p,
                                             _i32p, ctypes.POINTER(_int), _i32p, ctypes.POINTER(_int)]
            _lib = lib
    return _lib


def _p(a: np.ndarray, ptype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ptype)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


class OracleError(RuntimeError):
    pass


def decode_attention(q, k_cache, v_cache, block_table, seq_lens, want_probs=False):
    """out[B][h_q][d] (fp64) and, if asked, probs[B][h_q][max L]."""
    q, k_cache, v_cache = _f32(q), _f32(k_cache), _f32(v_cache)
    block_table, seq_lens = _i32(block_table), _i32(seq_lens)
    B, h_q, d = q.shape
    _, b, h_kv, d2 = k_cache.shape
    assert d2 == d
    out = np.zeros((B, h_q, d), dtype=np.float64)
    Lmax = int(seq_lens.max()) if B else 1
    probs = np.zeros((B, h_q, Lmax), dtype=np.float64) if want_probs else None
    rc = _load().orc_decode_attention(B, h_q, h_kv, d, b, _p(q, _f32p), _p(k_cache, _f32p),
                                      _p(v_cache, _f32p), _p(block_table, _i32p),
                                      block_table.shape[1], _p(seq_lens, _i32p), _p(out, _f64p),
                                      _p(probs, _f64p) if probs is not None else None,
                                      Lmax)
    if rc:
        raise OracleError("orc_decode_attention: %d" % rc)
    return (out, probs) if want_probs else out


def accumulate_window_score(probs, block_table, seq_lens, h_kv, b, w, score):
    """Update the paged window score ``score`` [N_total][b][h_kv] (fp64) in place."""
    probs, block_table, seq_lens = _f64(probs), _i32(block_table), _i32(seq_lens)
    assert score.dtype == np.float64 and score.flags["C_CONTIGUOUS"]
    B, h_q, stride = probs.shape
    rc = _load().orc_accumulate_window_score(B, h_q, h_kv, b, w, _p(block_table, _i32p),
                                             block_table.shape[1], _p(seq_lens, _i32p),
                                             _p(probs, _f64p), stride, _p(score, _f64p))
    if rc:
        raise OracleError("orc_accumulate_window_score: %d" % rc)
    return score


def window_score(q_window, k_cache, table_row, L, w):
    """Explicit observation-window score of one sequence: S[h_kv][L] (fp64)."""
    q_window, k_cache, table_row = _f32(q_window), _f32(k_cache), _i32(table_row)
    w_, h_q, d = q_window.shape
    assert w_ == w
    _, b, h_kv, _ = k_cache.shape
    S = np.zeros((h_kv, L), dtype=np.float64)
    rc = _load().orc_window_score(h_q, h_kv, d, b, w, _p(q_window, _f32p), _p(k_cache, _f32p),
                                  _p(table_row, _i32p), L, _p(S, _f64p))
    if rc:
        raise OracleError("orc_window_score: %d" % rc)
    return S


def global_score(S, F, table_row, b, first, alpha):
    """Alg. 2 on one sequence: S [h_kv][L] and paged F are updated in place."""
    assert S.dtype == np.float64 and F.dtype == np.float64
    assert S.flags["C_CONTIGUOUS"] and F.flags["C_CONTIGUOUS"]
    table_row = _i32(table_row)
    h_kv, L = S.shape
    rc = _load().orc_global_score(L, b, h_kv, int(bool(first)), float(alpha), _p(table_row, _i32p),
                                  _p(F, _f64p), _p(S, _f64p))
    if rc:
        raise OracleError("orc_global_score: %d" % rc)
    return S, F


def max_pool(x, kernel):
    x = _f64(x)
    y = np.empty_like(x)
    rc = _load().orc_max_pool(x.shape[0], int(kernel), _p(x, _f64p), _p(y, _f64p))
    if rc:
        raise OracleError("orc_max_pool: %d" % rc)
    return y


def redundancy(keys, b, p, tau, lightning):
    """R[L] for one (sequence, KV head) from its gathered keys [L][d]."""
    keys = _f32(keys)
    L, d = keys.shape
    R = np.empty(L, dtype=np.float64)
    rc = _load().orc_redundancy(L, d, b, _p(keys, _f32p), float(p), float(tau), int(bool(lightning)),
                                _p(R, _f64p))
    if rc:
        raise OracleError("orc_redundancy: %d" % rc)
    return R


def redundancy_rho(keys, b, p, lightning):
    """rho[L] (the row sums before normalisation) for one (sequence, KV head)."""
    keys = _f32(keys)
    L, d = keys.shape
    rho = np.empty(L, dtype=np.float64)
    rc = _load().orc_redundancy_rho(L, d, b, _p(keys, _f32p), float(p), int(bool(lightning)), _p(rho, _f64p))
    if rc:
        raise OracleError("orc_redundancy_rho: %d" % rc)
    return rho


def redundancy_rho_rows(keys, p, rows):
    """All-pairs rho at the given rows only (O(L) memory)."""
    keys = _f32(keys)
    L, d = keys.shape
    rows = _i32(rows)
    out = np.empty(rows.shape[0], dtype=np.float64)
    rc = _load().orc_redundancy_rho_rows(L, d, _p(keys, _f32p), float(p), _p(rows, _i32p), rows.shape[0],
                                         _p(out, _f64p))
    if rc:
        raise OracleError("orc_redundancy_rho_rows: %d" % rc)
    return out


def combine_and_window(S, w, lam, R=None):
    S = _f64(S).copy()
    Rr = _f64(R) if R is not None else None
    rc = _load().orc_combine_and_window(S.shape[0], int(w), float(lam),
                                        _p(Rr, _f64p) if Rr is not None else None, _p(S, _f64p))
    if rc:
        raise OracleError("orc_combine_and_window: %d" % rc)
    return S


def topk_keep(scores, k):
    """Ascending keep positions (padded with -1 to k), the 0/1 tag, the count."""
    scores = _f64(scores)
    L = scores.shape[0]
    keep = np.full(max(k, 1), -1, dtype=np.int32)
    tag = np.zeros(max(L, 1), dtype=np.uint8)
    n = _load().orc_topk_keep(L, int(k), _p(scores, _f64p), _p(keep, _i32p), _p(tag, _u8p))
    if n < 0:
        raise OracleError("orc_topk_keep failed")
    return keep[:k], tag[:L], n


def compact_alg4(base: np.ndarray, row_bytes, b, h_kv, kvh, src_table, dst_table, tag):
    """Alg. 4 byte move on a C-contiguous array viewed as bytes (in place)."""
    assert base.flags["C_CONTIGUOUS"]
    raw = base.reshape(-1).view(np.uint8)
    src_table, dst_table = _i32(src_table), _i32(dst_table)
    N = src_table.shape[0]
    full_tag = np.zeros(N * b, dtype=np.uint8)
    tag = np.asarray(tag, dtype=np.uint8)
    full_tag[: len(tag)] = tag
    return _load().orc_compact_alg4(_p(raw, _u8p), int(row_bytes), b, h_kv, kvh,
                                    _p(src_table, _i32p), N, _p(dst_table, _i32p),
                                    _p(full_tag, _u8p))


def needs_compression(L, b, N_max):
    return bool(_load().orc_needs_compression(int(L), int(b), int(N_max)))


def plan_targets(table, N_max, ref, fresh):
    table, ref, fresh = _i32(table), _i32(ref), _i32(fresh)
    N = table.shape[0]
    targets = np.zeros(max(N_max - 1, 1), dtype=np.int32)
    new_table = np.zeros(N_max, dtype=np.int32)
    released = np.zeros(N, dtype=np.int32)
    dropped = np.zeros(N, dtype=np.int32)
    nr, nd = _int(0), _int(0)
    fresh_buf = fresh if fresh.size else np.zeros(1, dtype=np.int32)
    used = _load().orc_plan_targets(_p(table, _i32p), N, N_max, _p(ref, _i32p),
                                    _p(fresh_buf, _i32p), int(fresh.size), _p(targets, _i32p),
                                    _p(new_table, _i32p), _p(released, _i32p), ctypes.byref(nr),
                                    _p(dropped, _i32p), ctypes.byref(nd))
    if used < 0:
        raise OracleError("orc_plan_targets failed")
    return {
        "targets": targets[: N_max - 1],
        "new_table": new_table,
        "released": released[: nr.value],
        "dropped_shared": dropped[: nd.value],
        "fresh_used": used,
    }
