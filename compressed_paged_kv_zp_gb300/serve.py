"""Serving loop on one GPU: the native request scheduler (zp_sched_*) drives
the libzp kernels over synthetic request traces, and the run reports
engine-level throughput -- tokens per second (TPS) and time per output token
(TPOT) as the Zipage paper defines them in §5.1.

Per step the scheduler [§4.3, §4.4] picks either a prefill step (admitted
requests) or a decode step (the running requests that can go on); then:
  * prefill: the prompt's keys and values are written into the request's
    blocks (synthetic values: prefill attention is not part of this path);
  * decode: per layer zp_append_kv + zp_paged_decode_attn, the window score
    accumulated into the request's query slot (a row of S) [§4.2];
  * compression of the triggered requests on a side stream with
    zp_compress_layers (per-request budgets, slot rows) [§4.1, §4.5, App. C.1];
    a compressing request sits out until its event has completed, then the
    scheduler swaps its table and releases what it dropped.
The model around attention (projections, MLP, sampling) is not simulated:
per-step inputs q, k, v are drawn on the device from a seeded generator.
"""
from __future__ import annotations

import argparse
import json
import time

import numpy as np
import torch

from . import (cache_desc, score_params, zp_append_kv, zp_compress_layers, zp_compress_workspace_size,
               zp_decode_workspace_size, zp_paged_decode_attn)
from .engine import upload
from .sched import CONSTRAINED, HYBRID, Scheduler


class ServeLoop:
    def __init__(self, h_q, h_kv, d, b, n_total, max_blocks, query_slots, table_stride, layers=1,
                 dtype=torch.bfloat16, window=None, params=None, policy=HYBRID, prefix_sharing=False,
                 max_running=256, max_prefill_tokens=16384, layer_stride=None, seed=0, device="cuda"):
        self.h_q, self.h_kv, self.d, self.b = h_q, h_kv, d, b
        self.n_total, self.N_max, self.M, self.stride, self.layers = n_total, max_blocks, query_slots, table_stride, layers
        self.window = window or b
        self.dtype = dtype
        self.dev = torch.device(device)
        self.desc = cache_desc(h_q, h_kv, d, b, n_total, dtype)
        self.params = params or score_params(window=self.window)
        self.layer_stride = max(1, min(layer_stride or layers, layers))
        self.sched = Scheduler(n_total, b, self.window, max_blocks, query_slots, policy=policy,
                               prefix_sharing=prefix_sharing, max_running=max_running,
                               max_prefill_tokens=max_prefill_tokens, table_stride=table_stride)
        self.K = torch.zeros(layers, n_total, b, h_kv, d, dtype=dtype, device=self.dev)
        self.V = torch.zeros_like(self.K)
        self.F = torch.zeros(layers, n_total, b, h_kv, dtype=torch.float32, device=self.dev)
        self.Lmax = table_stride * b
        # one score row per query slot and kv head [§4.2]
        self.S = torch.zeros(layers, query_slots, h_kv, self.Lmax, dtype=torch.float32, device=self.dev)
        self.ws = torch.empty(zp_decode_workspace_size(self.desc, max_running, table_stride), dtype=torch.uint8,
                              device=self.dev)
        self.score_ws = torch.empty(
            max(zp_compress_workspace_size(self.desc, min(max_running, query_slots), self.Lmax, self.layer_stride), 1),
            dtype=torch.uint8, device=self.dev)
        self.gen = torch.Generator(device=self.dev)
        self.gen.manual_seed(seed)
        self.side = torch.cuda.Stream(device=self.dev, priority=-1)  # compression kernels first when SMs free up
        self.inflight = []  # (done event, ids)
        self.budget = {}
        self.out = None
        self.last_step = None   # (kind, ids, inputs, tables) of the last step, for inspection
        self.last_keep = None   # (ids, keep [layers][n][h_kv][k]) of the last compressions
        self.events = []        # (step index, end event)
        self.first_step, self.last_step_of, self.n_out = {}, {}, {}
        self.stats = dict(prefill=0, decode=0, idle=0, compressions=0, preemptions=0, blocked=0)

    def add_request(self, rid, prompt_len, output_len, group=-1, prefix_len=0, max_blocks=0):
        self.sched.add(rid, prompt_len, output_len, group, prefix_len, max_blocks)
        self.budget[rid] = max_blocks or self.N_max
        self.n_out[rid] = output_len

    # ----------------------------------------------------------------- steps
    def _randn(self, *shape):
        return torch.randn(*shape, generator=self.gen, device=self.dev, dtype=torch.float32).to(self.dtype)

    def _prefill(self, st):
        b = self.b
        pos, blk = [], []
        for i in range(len(st["ids"])):
            p = np.arange(int(st["start"][i]), int(st["lens"][i]))
            pos.append(p)
            blk.append(st["tables"][i][p // b] * b + p % b)
        phys = upload(np.concatenate(blk).astype(np.int64), self.dev)
        n = int(phys.numel())
        if n:
            kf = self.K.view(self.layers, -1, self.h_kv, self.d)
            vf = self.V.view(self.layers, -1, self.h_kv, self.d)
            kf[:, phys] = self._randn(self.layers, n, self.h_kv, self.d)
            vf[:, phys] = self._randn(self.layers, n, self.h_kv, self.d)
        self.last_step = ("prefill", st["ids"], None, st["tables"])

    def _decode(self, st):
        B = len(st["ids"])
        table = upload(st["tables"], self.dev)
        lens = upload(st["lens"], self.dev)
        rows = upload(st["slots"], self.dev)
        q = self._randn(self.layers, B, self.h_q, self.d)
        kn = self._randn(self.layers, B, self.h_kv, self.d)
        vn = self._randn(self.layers, B, self.h_kv, self.d)
        out = torch.empty(self.layers, B, self.h_q, self.d, dtype=self.dtype, device=self.dev)
        for l in range(self.layers):
            zp_append_kv(self.desc, kn[l], vn[l], self.K[l], self.V[l], table, lens)
            zp_paged_decode_attn(self.desc, q[l], self.K[l], self.V[l], table, lens, out[l], score_accum=self.S[l],
                                 window=self.window, workspace=self.ws, score_rows=rows)
        self.out = out
        self.last_step = ("decode", st["ids"], (q, kn, vn), st["tables"])

    def _compress(self, comp):
        n = len(comp["ids"])
        if not n:
            return
        dev = self.dev
        tables = upload(comp["tables"], dev)
        lens = upload(comp["lens"], dev)
        first = upload(comp["first"].astype(np.uint8), dev)
        rows = upload(comp["slots"], dev)
        targets = upload(comp["targets"], dev)
        uniform = bool((comp["k"] == (self.N_max - 1) * self.b).all())
        k_seq = None if uniform else upload(comp["k"], dev)
        k = (self.N_max - 1) * self.b
        main = torch.cuda.current_stream(dev)
        ready = torch.cuda.Event()
        ready.record(main)
        with torch.cuda.stream(self.side):
            self.side.wait_event(ready)
            keep = torch.empty(self.layers, n, self.h_kv, k, dtype=torch.int32, device=dev)
            for l0 in range(0, self.layers, self.layer_stride):
                l1 = min(l0 + self.layer_stride, self.layers)
                zp_compress_layers(self.desc, self.params, self.K[l0:l1], self.V[l0:l1], tables, lens, first,
                                   self.S[l0:l1], self.F[l0:l1], targets, k, keep[l0:l1], self.Lmax, rows=rows,
                                   workspace=self.score_ws, k_seq=k_seq)
            done = torch.cuda.Event()
            done.record(self.side)
        for t in (tables, lens, first, rows, targets) + ((k_seq,) if k_seq is not None else ()):
            t.record_stream(self.side)
        self.inflight.append((done, comp["ids"].tolist()))
        self.last_keep = (comp["ids"].tolist(), keep)
        self.stats["compressions"] += n

    def _retire(self, block=False):
        still = []
        for done, ids in self.inflight:
            if block:
                done.synchronize()
            elif not done.query():
                still.append((done, ids))
                continue
            for rid in ids:
                self.sched.compression_done(rid)
        self.inflight = still

    def step(self):
        """One scheduler step; returns its kind ('prefill', 'decode', 'idle')."""
        self._retire()
        st = self.sched.schedule()
        kind = st["kind"]
        self.stats["preemptions"] += len(st["preempted"])
        self.stats["blocked"] += st["blocked"]
        self._compress(self.sched.take_compressions())  # retried compressions
        if kind == "prefill":
            self._prefill(st)
        elif kind == "decode":
            self._decode(st)
        else:
            self.last_step = ("idle", [], None, None)
            if self.inflight:
                self.inflight[0][0].synchronize()
        idx = len(self.events)
        ev = torch.cuda.Event(enable_timing=True)
        ev.record()
        self.events.append(ev)
        fin, pre = self.sched.commit()
        self.stats["preemptions"] += len(pre)
        self.stats[kind] += 1
        if kind != "idle":
            for rid in st["ids"].tolist():
                self.first_step.setdefault(rid, idx)
                self.last_step_of[rid] = idx
        self._compress(self.sched.take_compressions())
        return kind, fin

    def run(self, max_steps=10 ** 7):
        """Runs until every request has finished; returns the metrics."""
        t0 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        t0.record()
        for _ in range(max_steps):
            c = self.sched.counts()
            if c["waiting"] == 0 and c["running"] == 0:
                break
            self.step()
        else:
            raise RuntimeError("requests left after %d steps" % max_steps)
        self._retire(block=True)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        return self.metrics(t0, wall)

    def metrics(self, t0, wall):
        ends = [t0.elapsed_time(e) for e in self.events]  # ms since the start
        tokens = sum(self.n_out.values())
        total_ms = max(ends) if ends else 0.0
        tpot = []
        for rid, n in self.n_out.items():
            if n > 1 and rid in self.first_step:
                # first token at the end of its (last) prefill, last at the end of its last decode
                tpot.append((ends[self.last_step_of[rid]] - ends[self.first_step[rid]]) / (n - 1))
        return dict(tps=tokens / (total_ms / 1e3) if total_ms else 0.0, tokens=tokens, device_ms=total_ms,
                    wall_s=wall, tpot_ms_mean=float(np.mean(tpot)) if tpot else 0.0,
                    tpot_ms_p90=float(np.percentile(tpot, 90)) if tpot else 0.0, **self.stats)


def synthetic_trace(n, seed, prompt=(64, 512), output=(512, 4096), prefix_groups=0, prefix_len=0, budgets=None):
    """Requests with prompt and output lengths uniform in the given ranges
    (reasoning-style: short prompts, long outputs), optionally in prefix
    groups sharing prefix_len tokens, optionally with per-request budgets
    drawn uniformly from the range `budgets`."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        P = int(rng.integers(prompt[0], prompt[1] + 1))
        O = int(rng.integers(output[0], output[1] + 1))
        g, pl = -1, 0
        if prefix_groups and prefix_len <= P:
            g, pl = int(rng.integers(0, prefix_groups)), prefix_len
        nb = int(rng.integers(budgets[0], budgets[1] + 1)) if budgets else 0
        out.append((i, P, O, g, pl, nb))
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description="engine-level throughput of the scheduler + kernels on a synthetic trace")
    ap.add_argument("--policy", choices=["constrained", "hybrid"], default="hybrid")
    ap.add_argument("--prefix-sharing", action="store_true")
    ap.add_argument("--requests", type=int, default=256)
    ap.add_argument("--prompt", type=int, nargs=2, default=[64, 512])
    ap.add_argument("--output", type=int, nargs=2, default=[512, 4096])
    ap.add_argument("--prefix-groups", type=int, default=0)
    ap.add_argument("--prefix-len", type=int, default=0)
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--max-blocks", type=int, default=64)
    ap.add_argument("--query-slots", type=int, default=64)
    ap.add_argument("--blocks", type=int, default=16384)
    ap.add_argument("--max-running", type=int, default=256)
    ap.add_argument("--seed", type=int, default=0)
    a = ap.parse_args(argv)
    h_q, h_kv, d, b = 32, 8, 128, 16
    stride = (a.prompt[1] + a.output[1]) // b + 2
    loop = ServeLoop(h_q, h_kv, d, b, a.blocks, a.max_blocks, a.query_slots, stride, layers=a.layers,
                     policy=CONSTRAINED if a.policy == "constrained" else HYBRID, prefix_sharing=a.prefix_sharing,
                     max_running=a.max_running, seed=a.seed)
    for r in synthetic_trace(a.requests, a.seed, tuple(a.prompt), tuple(a.output), a.prefix_groups, a.prefix_len):
        loop.add_request(*r)
    m = loop.run()
    m.update(policy=a.policy, prefix_sharing=a.prefix_sharing, requests=a.requests, layers=a.layers,
             heads="%dq/%dkv" % (h_q, h_kv), head_dim=d, block=b, max_blocks=a.max_blocks, query_slots=a.query_slots,
             blocks=a.blocks, prompt=a.prompt, output=a.output)
    print(json.dumps(m))


if __name__ == "__main__":
    main()
