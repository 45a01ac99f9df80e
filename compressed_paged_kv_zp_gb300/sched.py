"""Binding of the request scheduler (include/zp_sched.h): constrained and
hybrid scheduling with query slots, preemption and prefix sharing [Zipage
§4.1, §4.3, §4.4, §4.5, Fig. 2].  Marshalling only; every decision is made
by libzp's scheduler.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import Pool, ZPError, _check, lib

CONSTRAINED, HYBRID = 0, 1
STEP_KIND = {0: "idle", 1: "prefill", 2: "decode"}
WAITING, RUNNING, COMPRESSING, FINISHED = 0, 1, 2, 3

_P = ctypes.c_void_p
_I32 = ctypes.c_int32


class SchedConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("block_size", "window", "max_blocks", "query_slots", "policy",
                                              "prefix_sharing", "max_running", "max_prefill_tokens",
                                              "table_stride")]


class _Step(ctypes.Structure):
    _fields_ = [("kind", _I32), ("n", _I32), ("n_preempted", _I32), ("n_blocked", _I32),
                ("ids", _P), ("lens", _P), ("start", _P), ("slots", _P), ("tables", _P), ("preempted", _P)]


class _Compressions(ctypes.Structure):
    _fields_ = [("n", _I32), ("ids", _P), ("lens", _P), ("slots", _P), ("k", _P), ("first", _P),
                ("tables", _P), ("targets", _P)]


lib.zp_sched_create.restype = _P
lib.zp_sched_create.argtypes = [ctypes.POINTER(SchedConfig), _P]
lib.zp_sched_destroy.argtypes = [_P]
lib.zp_sched_add_request.argtypes = [_P, _I32, _I32, _I32, _I32, _I32, _I32]
lib.zp_sched_schedule.argtypes = [_P, ctypes.POINTER(_Step)]
lib.zp_sched_commit.argtypes = [_P, _P, _P, _P, _P]
lib.zp_sched_take_compressions.argtypes = [_P, ctypes.POINTER(_Compressions)]
lib.zp_sched_compression_done.argtypes = [_P, _I32]
lib.zp_sched_counts.argtypes = [_P, _P]
lib.zp_sched_request_info.argtypes = [_P, _I32, _P]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_P)


class Scheduler:
    """Host scheduler over a block pool of n_total blocks (owned here)."""

    def __init__(self, n_total, block_size, window, max_blocks, query_slots, policy=HYBRID, prefix_sharing=False,
                 max_running=256, max_prefill_tokens=16384, table_stride=None, pool=None):
        self.pool = pool or Pool(n_total)
        stride = table_stride or max_blocks
        self.cfg = SchedConfig(int(block_size), int(window), int(max_blocks), int(query_slots), int(policy),
                               int(bool(prefix_sharing)), int(max_running), int(max_prefill_tokens), int(stride))
        self._s = lib.zp_sched_create(ctypes.byref(self.cfg), self.pool._p)
        if not self._s:
            raise ZPError(1, lib.zp_last_error().decode())
        cap, self.stride, self.N_max = int(max_running), int(stride), int(max_blocks)
        self._buf = {k: np.zeros(cap, np.int32) for k in ("ids", "lens", "start", "slots", "preempted", "fin",
                                                           "pre", "cids", "clens", "cslots", "ck", "cfirst")}
        self._tables = np.zeros((cap, stride), np.int32)
        self._ctables = np.zeros((cap, stride), np.int32)
        self._targets = np.zeros((cap, max(max_blocks - 1, 1)), np.int32)
        b = self._buf
        self._step = _Step(0, 0, 0, 0, _ptr(b["ids"]), _ptr(b["lens"]), _ptr(b["start"]), _ptr(b["slots"]),
                           _ptr(self._tables), _ptr(b["preempted"]))
        self._comp = _Compressions(0, _ptr(b["cids"]), _ptr(b["clens"]), _ptr(b["cslots"]), _ptr(b["ck"]),
                                   _ptr(b["cfirst"]), _ptr(self._ctables), _ptr(self._targets))

    def __del__(self):
        s = getattr(self, "_s", None)
        if s:
            lib.zp_sched_destroy(s)
            self._s = None

    def add(self, rid, prompt_len, output_len, group=-1, prefix_len=0, max_blocks=0):
        _check(lib.zp_sched_add_request(self._s, int(rid), int(prompt_len), int(output_len), int(group),
                                        int(prefix_len), int(max_blocks)))

    def schedule(self, copy=True):
        """The next step as a dict of numpy arrays (ids, lens, start, slots,
        tables [n][table_stride]) plus kind, preempted ids and n_blocked."""
        _check(lib.zp_sched_schedule(self._s, ctypes.byref(self._step)))
        st, b = self._step, self._buf
        n, npre = st.n, st.n_preempted
        cp = (lambda a: a.copy()) if copy else (lambda a: a)  # noqa: E731
        return dict(kind=STEP_KIND[st.kind], ids=cp(b["ids"][:n]), lens=cp(b["lens"][:n]), start=cp(b["start"][:n]),
                    slots=cp(b["slots"][:n]), tables=cp(self._tables[:n]), preempted=b["preempted"][:npre].tolist(),
                    blocked=int(st.n_blocked))

    def commit(self):
        """(finished ids, preempted ids) of the last step."""
        nf, npre = _I32(0), _I32(0)
        b = self._buf
        _check(lib.zp_sched_commit(self._s, _ptr(b["fin"]), ctypes.byref(nf), _ptr(b["pre"]), ctypes.byref(npre)))
        return b["fin"][: nf.value].tolist(), b["pre"][: npre.value].tolist()

    def take_compressions(self):
        """Compressions planned since the last call, as a dict of arrays."""
        _check(lib.zp_sched_take_compressions(self._s, ctypes.byref(self._comp)))
        n, b = self._comp.n, self._buf
        return dict(ids=b["cids"][:n].copy(), lens=b["clens"][:n].copy(), slots=b["cslots"][:n].copy(),
                    k=b["ck"][:n].copy(), first=b["cfirst"][:n].copy(), tables=self._ctables[:n].copy(),
                    targets=self._targets[:n, : self.N_max - 1].copy())

    def compression_done(self, rid):
        _check(lib.zp_sched_compression_done(self._s, int(rid)))

    def counts(self):
        out = np.zeros(5, np.int32)
        _check(lib.zp_sched_counts(self._s, _ptr(out)))
        return dict(zip(("waiting", "running", "finished", "free_slots", "free_blocks"), out.tolist()))

    def info(self, rid):
        out = np.zeros(7, np.int32)
        _check(lib.zp_sched_request_info(self._s, int(rid), _ptr(out)))
        keys = ("state", "L", "generated", "slot", "preemptions", "compressed", "n_blocks")
        d = dict(zip(keys, out.tolist()))
        d["compressed"] = bool(d["compressed"])
        return d
