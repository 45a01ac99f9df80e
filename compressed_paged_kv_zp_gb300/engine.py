"""Multi-step decode with Compressed PagedAttention on one GPU.

The host side of the hot path around the libzp kernels:
  * block allocation as sequences grow (Zipage paper §3);
  * the compression trigger after every step: N >= N_max blocks and the last
    block full (§4.1), with N_max optionally set per request (a budget of its
    own, at most the loop's N_max);
  * target blocks from the reference-counted pool, one planner call for all
    triggered sequences (§4.4);
  * the decode of the step in which a sequence triggers also forms the
    lightning redundancy row sums of its blocks from the keys it reads (no
    second read of the keys for the compression), when the library's
    one-kernel compression covers the cache and switches;
  * scoring, top-k and compaction on a side stream, ordered after the decode
    that produced the window score by a CUDA event (§4.5); in asynchronous
    mode the compressing sequences sit out decode until their event has
    completed, then rejoin with their new block table, while everybody else
    keeps decoding;
  * the blocks a compressed sequence no longer holds go back to the pool only
    after the compaction that reads them has completed.
All device work is libzp calls; torch provides memory, streams and events.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (Pool, cache_desc, score_params, zp_append_kv, zp_compress_layers, zp_compress_rho_supported,
               zp_compress_workspace_size, zp_needs_compression_batch, zp_decode_workspace_size,
               zp_paged_decode_attn)


def upload(arr: np.ndarray, dev) -> torch.Tensor:
    """Host array -> new device tensor without blocking the host: the values
    are staged in pinned memory (torch's caching host allocator keeps that
    block until the copy has completed) and copied on the current stream."""
    return torch.from_numpy(np.ascontiguousarray(arr)).pin_memory().to(dev, non_blocking=True)


def upload_packed(arrays, dev):
    """Several small host arrays -> device tensors of the same dtypes and
    shapes, through ONE pinned staging buffer and one copy (each array starts
    on a 16-byte boundary)."""
    offs, total = [], 0
    for a in arrays:
        offs.append(total)
        total += (a.nbytes + 15) // 16 * 16
    host = np.empty(max(total, 16), dtype=np.uint8)
    for a, o in zip(arrays, offs):
        host[o:o + a.nbytes] = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
    buf = torch.from_numpy(host).pin_memory().to(dev, non_blocking=True)
    out = []
    for a, o in zip(arrays, offs):
        dt = {np.dtype(np.int32): torch.int32, np.dtype(np.uint8): torch.uint8}[a.dtype]
        out.append(buf[o:o + a.nbytes].view(dt).view(a.shape))
    return out


class DecodeLoop:
    """Batch of sequences decoding over `layers` paged layers of one pool."""

    def __init__(self, h_q, h_kv, d, b, n_total, max_blocks, table_stride, layers=1, dtype=torch.bfloat16,
                 window=None, params=None, async_compress=False, layer_stride=None, device="cuda",
                 decode_rho=True):
        self.h_q, self.h_kv, self.d, self.b = h_q, h_kv, d, b
        self.n_total, self.N_max, self.stride, self.layers = n_total, max_blocks, table_stride, layers
        self.k = (max_blocks - 1) * b
        self.window = window or b
        self.dtype = dtype
        self.dev = torch.device(device)
        self.desc = cache_desc(h_q, h_kv, d, b, n_total, dtype)
        self.params = params or score_params(window=self.window)
        self.async_compress = async_compress
        self.decode_rho = decode_rho
        # layers compressed per call (App. C.1's layer stride): bounds the
        # scoring scratch to layer_stride layers
        self.layer_stride = max(1, min(layer_stride or layers, layers))
        self.K = torch.zeros(layers, n_total, b, h_kv, d, dtype=dtype, device=self.dev)
        self.V = torch.zeros_like(self.K)
        # global score cache F: paged like K (it moves with the kept tokens)
        self.F = torch.zeros(layers, n_total, b, h_kv, dtype=torch.float32, device=self.dev)
        self.pool = Pool(n_total)
        # compression stream at high priority: its CTAs are scheduled as soon
        # as SMs free up between decode launches, so a compressing sequence
        # sits out as few steps as possible
        self.side = torch.cuda.Stream(device=self.dev, priority=-1)
        self.B = 0
        self.compressions = 0
        self.pending = []  # (event, seqs, plan) of compressions in flight
        # buffers of the decode's row sums: reused once the compression that
        # read them has completed, so that no step allocates device or pinned
        # memory while the host runs ahead of the GPU
        self._rho_ring = []

    # ------------------------------------------------------------------ setup
    def add_sequences(self, lens, tables=None, max_blocks=None):
        """Register B sequences with `lens` cached tokens.  Their blocks come
        from the pool (lowest ids first) unless `tables` (np int32 [B][stride],
        already holding the sequences' block ids) is given; the caller fills
        the cache rows of those tokens directly (prefill is out of scope).
        max_blocks: optional per-request block budgets N_i in [2, N_max]; a
        request then compresses at N_i blocks to (N_i - 1) b tokens."""
        lens = np.asarray(lens, dtype=np.int32)
        B = len(lens)
        if max_blocks is None:
            self.N_seq = np.full(B, self.N_max, dtype=np.int32)
        else:
            self.N_seq = np.asarray(max_blocks, dtype=np.int32).copy()
            if self.N_seq.shape != (B,) or self.N_seq.min() < 2 or self.N_seq.max() > self.N_max:
                raise ValueError("max_blocks: one budget in [2, N_max] per sequence")
        self.uniform = bool((self.N_seq == self.N_max).all())
        self.B = B
        self._rho_ring = []  # slot maps are [B]
        self.lens = lens.copy()
        self.table = np.full((B, self.stride), -1, dtype=np.int32)
        if tables is None:
            for s in range(B):
                nb = (int(lens[s]) + self.b - 1) // self.b
                self.table[s, :nb] = self.pool.alloc(nb)
        else:
            self.table[:] = tables
            held = np.asarray(tables, dtype=np.int64).ravel()
            held = held[held >= 0]
            refs = np.bincount(held, minlength=self.n_total)
            self.pool.alloc(self.n_total)  # take every block, then give back the unused ones
            self.pool.release(np.nonzero(refs == 0)[0].tolist())
            extra = np.repeat(np.arange(self.n_total), np.maximum(refs - 1, 0))
            if len(extra):  # shared prefix blocks: one reference per holder
                self.pool.incref(extra.tolist())
        self.first = np.ones(B, dtype=np.uint8)  # never compressed yet
        self.active = np.ones(B, dtype=bool)
        self.table_dev = torch.from_numpy(self.table).to(self.dev)
        # attention score S: one row per (sequence, kv head), indexed by token
        # position, so sequences sharing prefix blocks keep their own scores
        self.S = torch.zeros(self.layers, B, self.h_kv, self.stride * self.b, dtype=torch.float32,
                             device=self.dev)
        self.ws = torch.empty(zp_decode_workspace_size(self.desc, B, self.stride), dtype=torch.uint8,
                              device=self.dev)
        Lmax = self.stride * self.b
        self.Lmax = Lmax
        self.use_rho = bool(self.decode_rho and zp_compress_rho_supported(self.desc, self.params, Lmax, self.k))
        self.score_ws = None if self.use_rho else torch.empty(
            max(zp_compress_workspace_size(self.desc, B, Lmax, self.layer_stride), 1), dtype=torch.uint8,
            device=self.dev)
        self.out = torch.zeros(self.layers, B, self.h_q, self.d, dtype=self.dtype, device=self.dev)

    def layer_stride(self):
        return self.n_total * self.b * self.h_kv * self.d

    # ------------------------------------------------------------------ step
    def step(self, q, k_new, v_new):
        """One decode step: q [layers][B][h_q][d], k_new/v_new [layers][B][h_kv][d].
        Returns the indices of the sequences that started a compression."""
        self._retire(block=not self.async_compress)
        act = self.active
        # grow: a sequence whose next token opens a block takes one from the
        # pool (a compressed sequence already holds its reserved block there);
        # blocks go out in sequence order, lowest free id first
        idx = np.nonzero(act)[0]
        pos = self.lens[idx]
        col = pos // self.b
        need = idx[(pos % self.b == 0) & (self.table[idx, np.minimum(col, self.stride - 1)] < 0)]
        if len(need):
            if int(self.lens[need].max()) // self.b >= self.stride:
                raise RuntimeError("a sequence outgrew table_stride blocks")
            self.table[need, self.lens[need] // self.b] = self.pool.alloc(len(need))
        self.lens[act] += 1
        self.table_dev.copy_(torch.from_numpy(self.table).pin_memory(), non_blocking=True)
        step_lens = upload(np.where(act, self.lens, 0).astype(np.int32), self.dev)
        main = torch.cuda.current_stream(self.dev)
        # the sequences that compress after this step: their decode also forms
        # the lightning row sums (row i of rho for the i-th of them)
        trig = zp_needs_compression_batch(self.lens, self.b, self.N_max, active=act, max_blocks_seq=self.N_seq)
        rho, buf, extra = None, None, {}
        if len(trig) and self.use_rho:
            n, Lr = len(trig), int(self.lens[trig].max())
            buf = self._rho_buffer(self.layers * n * self.h_kv * Lr)
            slot = buf["host"].numpy()
            slot[:] = -1
            slot[trig] = np.arange(n, dtype=np.int32)
            buf["rows"].copy_(buf["host"], non_blocking=True)
            rho = buf["rho"][: self.layers * n * self.h_kv * Lr].view(self.layers, n, self.h_kv, Lr)
            extra = dict(rho_rows=buf["rows"], rho_threshold=self.params.threshold)
        for l in range(self.layers):
            zp_append_kv(self.desc, k_new[l], v_new[l], self.K[l], self.V[l], self.table_dev, step_lens)
            zp_paged_decode_attn(self.desc, q[l], self.K[l], self.V[l], self.table_dev, step_lens, self.out[l],
                                 score_accum=self.S[l], window=self.window, workspace=self.ws,
                                 rho=None if rho is None else rho[l], **extra)
        if len(trig):
            done = self._compress(trig, main, rho)
            if buf is not None:
                buf["busy"] = done
        return trig.tolist()

    def _rho_buffer(self, elems):
        """A free buffer of at least `elems` floats, with its slot-map arrays
        (device and pinned host int32 [B])."""
        for e in self._rho_ring:
            if e["rho"].numel() >= elems and (e["busy"] is None or e["busy"].query()):
                e["busy"] = None
                return e
        e = dict(rho=torch.empty(elems + elems // 4, dtype=torch.float32, device=self.dev),
                 rows=torch.empty(self.B, dtype=torch.int32, device=self.dev),
                 host=torch.empty(self.B, dtype=torch.int32).pin_memory(), busy=None)
        self._rho_ring.append(e)
        return e

    def _compress(self, seqs, main, rho=None):
        n = len(seqs)
        nb = (self.lens[seqs] // self.b).astype(np.int32)
        sub_tables = np.ascontiguousarray(self.table[seqs])
        plan = self.pool.plan_compaction_batch(sub_tables, nb, self.N_max,
                                               max_blocks_seq=None if self.uniform else self.N_seq[seqs])
        parts = [sub_tables, self.lens[seqs].astype(np.int32), seqs.astype(np.int32), plan["targets"],
                 self.first[seqs].astype(np.uint8)]
        if not self.uniform:
            parts.append(((self.N_seq[seqs] - 1) * self.b).astype(np.int32))
        dev_parts = upload_packed(parts, self.dev)
        tables_dev, lens_dev, rows_dev, targets_dev, first_dev = dev_parts[:5]
        k_seq = None if self.uniform else dev_parts[5]
        ready = torch.cuda.Event()
        ready.record(main)
        with torch.cuda.stream(self.side):
            self.side.wait_event(ready)
            keep = torch.empty(self.layers, n, self.h_kv, self.k, dtype=torch.int32, device=self.dev)
            for l0 in range(0, self.layers, self.layer_stride):  # scores, keep sets, moves of a layer group
                l1 = min(l0 + self.layer_stride, self.layers)
                zp_compress_layers(self.desc, self.params, self.K[l0:l1], self.V[l0:l1], tables_dev, lens_dev,
                                   first_dev, self.S[l0:l1], self.F[l0:l1], targets_dev, self.k, keep[l0:l1],
                                   self.Lmax, rows=rows_dev, workspace=self.score_ws, k_seq=k_seq,
                                   rho=None if rho is None else rho[l0:l1])
            done = torch.cuda.Event()
            done.record(self.side)
        tables_dev.record_stream(self.side)  # every part is a view of one device buffer
        self.active[seqs] = False
        self.last_keep = (seqs, keep)  # for inspection: [layers][n][h_kv][k]
        self.pending.append((done, seqs, plan, keep))
        self.compressions += n
        if not self.async_compress:
            main.wait_event(done)
        return done

    def _retire(self, block=False):
        """Apply the compressions that have finished: new tables, lengths and
        the release of the blocks the sequences dropped."""
        still = []
        for done, seqs, plan, keep in self.pending:
            if block:
                torch.cuda.current_stream(self.dev).wait_event(done)
            elif not done.query():
                still.append((done, seqs, plan, keep))
                continue
            for i, s in enumerate(seqs):
                self.table[s, :] = -1
                self.table[s, : self.N_max] = plan["new_tables"][i]
                self.lens[s] = (int(self.N_seq[s]) - 1) * self.b
                self.first[s] = 0
                self.active[s] = True
                nd = int(plan["n_dropped"][i])
                if nd:
                    self.pool.release(plan["dropped"][i, :nd].tolist())
        self.pending = still

    def drain(self):
        for done, _, _, _ in self.pending:
            done.synchronize()
        self._retire(block=True)

