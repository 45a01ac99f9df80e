"""The decode-with-compression loop on the oracle, for the multi-step GPU
tests: fp64 arithmetic, float32 caches holding the bf16 values the device
sees, and a Python mirror of the block pool with its own block ids.

Every step: grow the block table (lowest free block first), append the new
token, decode with window-score accumulation, apply the §4.1 trigger.  A
compression scores, ranks and compacts into the §4.4 targets, swaps the table
and releases the dropped blocks.  The loop can mirror any subset of a GPU
batch's sequences and layers (they are independent); block ids are its own,
so only outputs, keep sets and moved rows are compared with the device.
"""
import numpy as np

import oracle
from oracle import pipeline
from tests.gpu_util import keep_sets_match


class OracleLoop:
    def __init__(self, cfg, K, V, table, lens):
        """cfg: h_q, h_kv, d, b, N_max, w, layers, n_total.  K, V: float32
        [layers][n_total][b][h_kv][d]; table int32 [B][stride]; lens [B]."""
        self.c = cfg
        self.K, self.V = K.copy(), V.copy()
        self.S = np.zeros(K.shape[:-1])  # [layers][n_total][b][h_kv] fp64
        self.F = np.zeros(K.shape[:-1])
        self.table = table.copy()
        self.lens = lens.copy()
        self.first = np.ones(len(lens), dtype=bool)
        self.ref = np.zeros(cfg["n_total"], dtype=np.int32)
        for x in table.flatten():
            if x >= 0:
                self.ref[x] += 1

    @classmethod
    def mirror(cls, cfg, K_blocks, V_blocks, lens, stride, spare):
        """A loop over sequences whose cached rows are given block by block
        (K_blocks[s]: float32 [layers][n_blocks_s][b][h_kv][d]); their blocks
        are numbered consecutively, `spare` free blocks follow."""
        nb = [kb.shape[1] for kb in K_blocks]
        n_total = sum(nb) + spare
        layers = K_blocks[0].shape[0]
        shape = (layers, n_total) + K_blocks[0].shape[2:]
        K = np.zeros(shape, dtype=np.float32)
        V = np.zeros(shape, dtype=np.float32)
        table = np.full((len(nb), stride), -1, dtype=np.int32)
        cur = 0
        for s, n in enumerate(nb):
            K[:, cur:cur + n] = K_blocks[s]
            V[:, cur:cur + n] = V_blocks[s]
            table[s, :n] = np.arange(cur, cur + n)
            cur += n
        return cls(dict(cfg, n_total=n_total, layers=layers), K, V, table, np.asarray(lens, dtype=np.int32))

    def alloc(self):
        blk = int(np.nonzero(self.ref == 0)[0][0])
        self.ref[blk] = 1
        return blk

    def step(self, q, kn, vn):
        """q [layers][B][h_q][d], kn/vn [layers][B][h_kv][d] (float32).
        Returns the outputs [layers][B][h_q][d] and the triggered sequences."""
        c = self.c
        b = c["b"]
        for s in range(len(self.lens)):
            pos = int(self.lens[s])
            if pos % b == 0 and self.table[s, pos // b] < 0:
                self.table[s, pos // b] = self.alloc()
        self.lens += 1
        outs = []
        for l in range(c["layers"]):
            for s in range(len(self.lens)):
                P = int(self.lens[s]) - 1
                blk = self.table[s, P // b]
                self.K[l, blk, P % b] = kn[l, s]
                self.V[l, blk, P % b] = vn[l, s]
            out, probs = oracle.decode_attention(q[l], self.K[l], self.V[l], self.table, self.lens, want_probs=True)
            S = np.ascontiguousarray(self.S[l])
            oracle.accumulate_window_score(probs, self.table, self.lens, c["h_kv"], b, c["w"], S)
            self.S[l] = S
            outs.append(out)
        trig = [s for s in range(len(self.lens)) if oracle.needs_compression(int(self.lens[s]), b, c["N_max"])]
        return np.stack(outs), trig

    def compress(self, s, gpu_keep):
        """Scores and keep sets of sequence s on every layer against the
        device's keep sets gpu_keep [layers][h_kv][k]; returns the number of
        reported near-tie swaps.  The moves use the device's keep sets, so
        after a reported near-tie both sides stay in the same state."""
        c = self.c
        b, N_max = c["b"], c["N_max"]
        L = int(self.lens[s])
        k = (N_max - 1) * b
        N = L // b
        fresh = np.nonzero(self.ref == 0)[0].astype(np.int32)
        plan = oracle.plan_targets(self.table[s, :N], N_max, self.ref, fresh)
        for blk in plan["new_table"]:
            if self.ref[blk] == 0:
                self.ref[blk] = 1
        swaps = 0
        prm = pipeline.ScoreParams(window=c["w"])
        for l in range(c["layers"]):
            S_seq = pipeline.gather_slots(self.S[l], self.table[s], L, b)
            F = np.ascontiguousarray(self.F[l])
            sc = pipeline.final_scores(S_seq, self.K[l], F, self.table[s], L, b, bool(self.first[s]), prm)
            self.F[l] = F
            for h in range(c["h_kv"]):
                ref_keep = oracle.topk_keep(sc[h], k)[0]
                swaps += keep_sets_match(gpu_keep[l, h], ref_keep, sc[h], k, L)
        pipeline.compact_sequence([self.K, self.V, self.F], [c["d"] * 4, c["d"] * 4, 8], b, c["h_kv"],
                                  self.table[s], N, plan["targets"], gpu_keep, L)
        for blk in list(plan["released"]) + list(plan["dropped_shared"]):
            self.ref[blk] -= 1
        self.table[s, :] = -1
        self.table[s, :N_max] = plan["new_table"]
        self.lens[s] = k
        self.first[s] = False
        return swaps
