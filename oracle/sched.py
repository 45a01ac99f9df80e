"""Oracle of the request scheduler around Compressed PagedAttention (test
infrastructure, see ``oracle/__init__.py``).

Plain Python, one decision at a time, in the order the pages state the rules:

* Zipage §4.1: a request holds at most N_max blocks outside prefill; after a
  decode step, N >= N_max with the last block full triggers a compression
  that keeps N_max - 1 blocks and reserves one more; the rest is released.
* Zipage §4.2, §4.3 (query slots): only requests holding one of the M query
  slots can be compressed.
* Zipage §4.3, constrained scheduling: at most M requests run, each with a
  slot; a request that finds no free block is blocked, never preempted.
* Zipage §4.3, hybrid scheduling (and Fig. 2): requests are admitted when
  their prefill blocks are free, slot or not; only the first M requests of the
  running queue may hold slots, freed slots go to the foremost requests
  without one; a request without a slot may decode while it holds fewer than
  N_max blocks or its token falls before the last w positions of its block,
  and is blocked otherwise; a request that finds no free block preempts the
  last running request without a slot, and once none is left it is blocked as
  under constrained scheduling.
* Zipage §4.4 (shared prefix): blocks are reference counted, compaction of a
  request holding shared blocks goes to new target blocks, and with prefix
  sharing on, a request that finds no block (for decoding or for the targets
  of its compression) preempts the last uncompressed request, slot or not.
* Zipage §4.5: a compressing request sits out decode until its compression
  has completed; the others keep decoding.
* Zipage, Limitations: N_max may be an attribute of each request.

Readings where the pages leave a step open (plainest choice, also stated by
the product's header): prefill and decode are separate steps and waiting
requests are admitted first (first come, first served, no skipping); a
preempted request loses its cache and goes back to the front of the waiting
queue, its generated tokens become part of its prompt on re-admission (which
yields one more token); the first M positions rule is applied when slots are
handed out at the start of a step and after a step's finishes; victims of a
preemption during decode are taken from the back among the requests not yet
scanned in that step, then the scanning request itself; the trigger is
checked only for requests that decoded in the step.
"""
from __future__ import annotations

from collections import deque

import numpy as np

from . import plan_targets

CONSTRAINED, HYBRID = 0, 1
WAITING, RUNNING, COMPRESSING, FINISHED = 0, 1, 2, 3


class OracleSchedError(RuntimeError):
    pass


class _Req:
    def __init__(self, rid, P, O, group, prefix_len, N):
        self.id, self.P, self.O = rid, P, O
        self.group, self.prefix_len, self.N = group, prefix_len, N
        self.state = WAITING
        self.L = 0
        self.generated = 0
        self.slot = -1
        self.table = []
        self.compressed = False
        self.want_compress = False
        self.holds_prefix = False
        self.preemptions = 0


class Scheduler:
    def __init__(self, n_total, b, w, N_max, M, policy, prefix_sharing, max_running, max_prefill_tokens,
                 table_stride):
        self.n_total, self.b, self.w, self.N_max, self.M = n_total, b, w, N_max, M
        self.policy, self.sharing = policy, bool(prefix_sharing)
        self.max_running, self.max_prefill_tokens, self.stride = max_running, max_prefill_tokens, table_stride
        self.ref = np.zeros(n_total, dtype=np.int32)
        self.slot_used = [False] * M
        self.reqs = {}
        self.waiting = deque()
        self.running = []
        self.prefix = {}  # group -> [blocks, holders]
        self.group_len = {}  # group -> its prefix length
        self.started = []  # compressions planned and not yet taken
        self.last = None

    # ------------------------------------------------------------- helpers
    def _alloc(self, n):
        free = np.nonzero(self.ref == 0)[0][:n]
        if len(free) < n:
            raise OracleSchedError("pool exhausted")
        self.ref[free] = 1
        return [int(x) for x in free]

    def _num_free(self):
        return int((self.ref == 0).sum())

    def _release(self, blocks):
        for x in blocks:
            assert self.ref[x] > 0
            self.ref[x] -= 1

    def _leave_prefix(self, r):
        if r.holds_prefix:
            ent = self.prefix[r.group]
            ent[1] -= 1
            if ent[1] == 0:
                del self.prefix[r.group]
            r.holds_prefix = False

    def _free_slot(self, r):
        if r.slot >= 0:
            self.slot_used[r.slot] = False
            r.slot = -1

    def _assign_slots(self):
        for r in self.running[: self.M]:
            if r.slot < 0:
                free = [i for i, u in enumerate(self.slot_used) if not u]
                if not free:
                    return
                r.slot = free[0]
                self.slot_used[free[0]] = True

    def _victim_ok(self, v):
        if v.state != RUNNING or v.compressed:
            return False
        if self.sharing:
            return True
        return self.policy == HYBRID and v.slot < 0

    def _preempt(self, v):
        self._release(v.table)
        self._leave_prefix(v)
        self._free_slot(v)
        v.table, v.L = [], 0
        v.want_compress = False
        v.state = WAITING
        v.preemptions += 1
        self.running.remove(v)
        self.waiting.appendleft(v)
        return v.id

    def _finish(self, r):
        self._release(r.table)
        self._leave_prefix(r)
        self._free_slot(r)
        r.table = []
        r.state = FINISHED
        self.running.remove(r)

    def _try_compress(self, r, preempted):
        nb = r.L // self.b
        table = r.table[:nb]
        need = sum(1 for t in range(r.N) if self.ref[table[t]] > 1)
        while self._num_free() < need and self.sharing:
            victim = next((v for v in reversed(self.running) if self._victim_ok(v)), None)
            if victim is None:
                break
            preempted.append(self._preempt(victim))
            if victim is r:
                return
            need = sum(1 for t in range(r.N) if self.ref[table[t]] > 1)
        if self._num_free() < need:
            return  # stays triggered; tried again at the next step
        fresh = np.nonzero(self.ref == 0)[0][:need].astype(np.int32)
        plan = plan_targets(np.asarray(table, np.int32), r.N, self.ref.copy(), fresh)
        for x in fresh[: plan["fresh_used"]]:
            self.ref[x] = 1
        dropped = [int(x) for x in plan["released"]] + [int(x) for x in plan["dropped_shared"]]
        self._leave_prefix(r)
        self.started.append(dict(id=r.id, L=r.L, slot=r.slot, k=(r.N - 1) * self.b, first=not r.compressed,
                                 table=list(table), targets=[int(x) for x in plan["targets"]],
                                 new_table=[int(x) for x in plan["new_table"]], dropped=dropped))
        r.state = COMPRESSING
        r.want_compress = False

    # ------------------------------------------------------------- requests
    def add(self, rid, prompt_len, output_len, group=-1, prefix_len=0, max_blocks=0):
        N = max_blocks or self.N_max
        if rid in self.reqs or prompt_len < 1 or output_len < 1 or not 2 <= N <= self.N_max:
            raise OracleSchedError("bad request")
        if prefix_len % self.b or prefix_len > prompt_len or (prefix_len and group < 0):
            raise OracleSchedError("bad prefix")
        if prompt_len + output_len - 1 > self.stride * self.b:
            raise OracleSchedError("request longer than a block table")
        if prefix_len and self.group_len.setdefault(group, prefix_len) != prefix_len:
            raise OracleSchedError("a prefix group has one prefix length")
        r = _Req(rid, prompt_len, output_len, group, prefix_len, N)
        self.reqs[rid] = r
        self.waiting.append(r)

    def schedule(self):
        """The next step: dict(kind, ids, lens, start, slots, tables, preempted, blocked)."""
        preempted = []
        self._assign_slots()
        for r in list(self.running):
            if r.want_compress and r.state == RUNNING:
                self._try_compress(r, preempted)
        # ---- admission (prefill)
        admitted, tokens = [], 0
        while self.waiting:
            r = self.waiting[0]
            if len(self.running) >= self.max_running:
                break
            if self.policy == CONSTRAINED and len(self.running) >= self.M:
                break
            L = r.P + r.generated
            if admitted and tokens + L > self.max_prefill_tokens:
                break
            nb = -(-L // self.b)
            pb = r.prefix_len // self.b if self.sharing else 0
            cached = pb > 0 and r.group in self.prefix
            need = nb - pb if cached else nb
            if need > self._num_free():
                break
            self.waiting.popleft()
            if cached:
                pre = self.prefix[r.group]
                for x in pre[0]:
                    self.ref[x] += 1
                pre[1] += 1
                r.table = list(pre[0]) + self._alloc(need)
                r.holds_prefix = True
                start = r.prefix_len
            else:
                r.table = self._alloc(need)
                if pb > 0:
                    self.prefix[r.group] = [list(r.table[:pb]), 1]
                    r.holds_prefix = True
                start = 0
            r.L = L
            r.generated += 1
            r.state = RUNNING
            self.running.append(r)
            admitted.append((r, start))
            tokens += L
        if admitted:
            self._assign_slots()
            self.last = ("prefill", [r for r, _ in admitted])
            return dict(kind="prefill", ids=[r.id for r, _ in admitted], lens=[r.L for r, _ in admitted],
                        start=[s for _, s in admitted], slots=[r.slot for r, _ in admitted],
                        tables=[list(r.table) for r, _ in admitted], preempted=preempted, blocked=0)
        # ---- decode
        batch, blocked = [], 0
        idx = 0
        while idx < len(self.running):
            r = self.running[idx]
            if r.state != RUNNING:
                idx += 1
                continue
            if r.want_compress:
                blocked += 1
                idx += 1
                continue
            pos = r.L
            if r.slot < 0 and pos // self.b + 1 >= r.N and pos % self.b >= self.b - self.w:
                blocked += 1
                idx += 1
                continue
            col = pos // self.b
            if pos % self.b == 0 and col >= len(r.table):
                gone = False
                while self._num_free() == 0:
                    victim = next((v for v in reversed(self.running[idx + 1:]) if self._victim_ok(v)), None)
                    if victim is None and self._victim_ok(r):
                        victim = r
                    if victim is None:
                        break
                    preempted.append(self._preempt(victim))
                    if victim is r:
                        gone = True
                        break
                if gone:
                    continue
                if self._num_free() == 0:
                    blocked += 1
                    idx += 1
                    continue
                r.table += self._alloc(1)
            r.L += 1
            batch.append(r)
            idx += 1
        if not batch:
            busy = any(r.state == COMPRESSING for r in self.running) or bool(self.started)
            if not busy and (self.running or self.waiting):
                raise OracleSchedError("deadlock: nothing can run")
            self.last = ("idle", [])
            return dict(kind="idle", ids=[], lens=[], start=[], slots=[], tables=[], preempted=preempted,
                        blocked=blocked)
        self.last = ("decode", batch)
        return dict(kind="decode", ids=[r.id for r in batch], lens=[r.L for r in batch],
                    start=[r.L - 1 for r in batch], slots=[r.slot for r in batch],
                    tables=[list(r.table) for r in batch], preempted=preempted, blocked=blocked)

    def commit(self):
        """Apply the last step once its device work is issued; returns
        (finished ids, preempted ids)."""
        kind, reqs = self.last
        self.last = ("idle", [])
        finished, preempted = [], []
        if kind == "prefill":
            for r in reqs:
                if r.generated >= r.O:
                    finished.append(r.id)
                    self._finish(r)
        elif kind == "decode":
            for r in reqs:
                r.generated += 1
                if r.generated >= r.O:
                    finished.append(r.id)
                    self._finish(r)
                elif r.slot >= 0 and r.L % self.b == 0 and r.L // self.b >= r.N:
                    r.want_compress = True
            for r in reqs:
                if r.want_compress and r.state == RUNNING:
                    self._try_compress(r, preempted)
        self._assign_slots()
        return finished, preempted

    def take_compressions(self):
        out, self.started = self.started, []
        return out

    def compression_done(self, rid, plan):
        r = self.reqs[rid]
        assert r.state == COMPRESSING
        r.table = list(plan["new_table"])
        r.L = (r.N - 1) * self.b
        r.compressed = True
        r.state = RUNNING
        self._release(plan["dropped"])

    # ------------------------------------------------------------- queries
    def counts(self):
        return dict(waiting=len(self.waiting), running=len(self.running),
                    finished=sum(1 for r in self.reqs.values() if r.state == FINISHED),
                    free_slots=sum(1 for u in self.slot_used if not u), free_blocks=self._num_free())

    def info(self, rid):
        r = self.reqs[rid]
        return dict(state=r.state, L=r.L, generated=r.generated, slot=r.slot, preemptions=r.preemptions,
                    compressed=r.compressed, n_blocks=len(r.table))
