"""The compression pipeline of the oracle, composed in the paper's order.

Test infrastructure (see ``oracle/__init__.py``).  Every arithmetic step is a
call into ``zp_oracle.c``; this file only sequences the steps and gathers rows
through the block table.  Order of the steps, as the per-operation timing of
[Zipage App. C.7, Figs. 13/14] lists them: attention score -> global score ->
pooling -> redundancy score -> window mask -> top-k -> compress kv -> compress
score.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import (combine_and_window, compact_alg4, global_score, max_pool,
               plan_targets, redundancy, topk_keep)


@dataclasses.dataclass
class ScoreParams:
    """Scoring switches and constants.

    alpha, lam, tau: the recommended values of [Zipage App. C.8].
    pool_kernel and p: not given by the paper (parameters, unpinned defaults).
    pool_policy: 0 never, 1 first compression only (recommended, App. C.8),
    2 every compression.
    """
    window: int = 16
    use_global: bool = True
    alpha: float = 0.8
    pool_kernel: int = 7
    pool_policy: int = 1
    use_similarity: bool = True
    lightning: bool = True
    p: float = 0.9
    lam: float = 0.2
    tau: float = 0.4


def gather_rows(cache_layer: np.ndarray, table_row, L: int, b: int) -> np.ndarray:
    """[L][h_kv][...] logical rows of one sequence (a gather, no arithmetic)."""
    t = np.arange(L)
    blocks = np.asarray(table_row, dtype=np.int64)[t // b]
    return cache_layer[blocks, t % b]


def gather_slots(paged: np.ndarray, table_row, L: int, b: int) -> np.ndarray:
    """[h_kv][L] view of a per-slot array [N_total][b][h_kv] for one sequence."""
    return np.ascontiguousarray(gather_rows(paged, table_row, L, b).T)


def final_scores(S: np.ndarray, k_layer: np.ndarray, F: np.ndarray | None, table_row, L: int,
                 b: int, first: bool, prm: ScoreParams) -> np.ndarray:
    """Scores of one sequence, one layer, all KV heads, ready for the top-k.

    S: [h_kv][L] attention score (explicit window or accumulated).  F: paged
    global score cache of this layer, updated in place when use_global.
    k_layer: the layer's key cache [N_total][b][h_kv][d] (float32).
    """
    S = np.ascontiguousarray(S, dtype=np.float64).copy()
    h_kv = S.shape[0]
    if prm.use_global:
        assert F is not None
        global_score(S, F, table_row, b, first, prm.alpha)
    pool = prm.pool_kernel > 1 and (prm.pool_policy == 2 or (prm.pool_policy == 1 and first))
    out = np.empty_like(S)
    keys = gather_rows(k_layer, table_row, L, b) if prm.use_similarity else None
    for kvh in range(h_kv):
        s = max_pool(S[kvh], prm.pool_kernel) if pool else S[kvh]
        R = redundancy(keys[:, kvh, :], b, prm.p, prm.tau, prm.lightning) if prm.use_similarity else None
        out[kvh] = combine_and_window(s, prm.window, prm.lam, R)
    return out


def keep_sets(scores: np.ndarray, k: int) -> np.ndarray:
    """[h_kv][k] ascending keep positions (-1 padded) from [h_kv][L] scores."""
    return np.stack([topk_keep(scores[h], k)[0] for h in range(scores.shape[0])])


def compact_sequence(caches, row_bytes, b: int, h_kv: int, table_row, N: int, targets,
                     keep: np.ndarray, L: int) -> None:
    """Alg. 4 for every layer and KV head of one sequence.

    caches: list of (array, row_bytes) where array is [layers][N_total][b][h_kv][...]
    keep: [layers][h_kv][k] ascending positions.  Moves in place (numpy arrays).
    """
    src = np.asarray(table_row[:N], dtype=np.int32)
    dst = np.asarray(targets, dtype=np.int32)
    for arr, rb in zip(caches, row_bytes):
        for layer in range(arr.shape[0]):
            for kvh in range(h_kv):
                tag = np.zeros(N * b, dtype=np.uint8)
                kp = keep[layer][kvh]
                tag[kp[kp >= 0]] = 1
                compact_alg4(arr[layer], rb, b, h_kv, kvh, src, dst, tag[:L])


__all__ = ["ScoreParams", "gather_rows", "gather_slots", "final_scores", "keep_sets",
           "compact_sequence", "plan_targets"]
