"""Shared helpers of the GPU parity tests: move a seeded case to the device and
compare device results with the oracle at the documented tolerances."""
import numpy as np
import torch

import zp_inputs

# Tolerances (stated by the workload definition for this path):
#   attention outputs: bf16 inputs 2e-2 abs / 1e-2 rel; fp32 inputs 1e-4.
#   scores: computed in fp32 from the same inputs; checked at 1e-3 relative
#   (bf16) / 1e-4 relative (fp32), which is tighter than the output tolerance
#   because the scores decide integer keep sets.
TOL_OUT = {"bf16": dict(atol=2e-2, rtol=1e-2), "f32": dict(atol=1e-4, rtol=1e-4)}
TOL_SCORE = {"bf16": dict(atol=1e-8, rtol=1e-3), "f32": dict(atol=1e-9, rtol=1e-4)}
TIE_REL = 1e-5


class DeviceCase:
    def __init__(self, case: zp_inputs.PagedCase, dev="cuda"):
        self.c = case
        self.q = case.q.to(dev)
        self.K = case.k_cache.contiguous().to(dev)  # [layers][N_total][b][h_kv][d]
        self.V = case.v_cache.contiguous().to(dev)
        self.table = case.block_table.to(dev)
        self.lens = case.seq_lens.to(dev)

    def np_k(self, layer=0):
        return self.K[layer].float().cpu().numpy()

    def np_v(self, layer=0):
        return self.V[layer].float().cpu().numpy()


def gather_slots(paged, table_row, L, b):
    t = np.arange(L)
    return np.ascontiguousarray(paged[np.asarray(table_row)[t // b], t % b].T)


def keep_sets_match(got, ref, scores_ref, k, L):
    """Index sets equal except for swaps among oracle scores within TIE_REL of
    the k-th score; returns the number of such swaps (reported)."""
    got = set(int(x) for x in got if x >= 0)
    ref = set(int(x) for x in ref if x >= 0)
    if got == ref:
        return 0
    if L <= k:
        raise AssertionError("under budget the keep set must be everything")
    s = np.asarray(scores_ref, dtype=np.float64)[:L]
    kth = np.sort(s)[::-1][k - 1]
    diff = got ^ ref
    for t in diff:
        if not (abs(s[t] - kth) <= TIE_REL * max(abs(kth), 1e-30) or (np.isinf(s[t]) and np.isinf(kth))):
            raise AssertionError("position %d (score %r, k-th %r) differs beyond ties" % (t, s[t], kth))
    assert len(got) == len(ref)
    return len(diff) // 2
