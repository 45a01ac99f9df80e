"""The request scheduler of libzp (include/zp_sched.h) against the scheduler
oracle: identical decisions, step by step, on seeded random request traces
(prompt and output lengths, long prompts beyond the budget, shared prefixes,
per-request budgets), with the pool tight enough that requests block, get
preempted and wait for slots; compressions complete after random delays,
given to both sides alike.  Every step also checks the invariants the pages
state: at most M slots, distinct; constrained scheduling runs at most M
requests, all with slots, and without prefix sharing never preempts; a
window token is decoded only with a slot; a compressed request is never
preempted and holds at most its budget of blocks; every request ends with
exactly its output length.  No GPU is used.
"""
import numpy as np
import pytest

from oracle.sched import OracleSchedError
from oracle.sched import Scheduler as OracleScheduler

CASES = [
    # name, policy, sharing, budgets, M, n_total
    ("constrained", 0, False, False, 4, 60),
    ("hybrid", 1, False, False, 2, 60),
    ("hybrid_tight", 1, False, False, 1, 40),
    ("constrained_prefix", 0, True, False, 3, 70),
    ("hybrid_prefix", 1, True, False, 2, 70),
    ("hybrid_budgets", 1, False, True, 3, 60),
    ("hybrid_prefix_budgets", 1, True, True, 2, 80),
]


def _trace(rng, n, b, N_max, stride, sharing, budgets):
    reqs = []
    group_len = {g: int(rng.integers(1, 4)) * b for g in range(3)}
    for i in range(n):
        P = int(rng.choice([rng.integers(1, 3 * b), rng.integers(3 * b, 2 * N_max * b)]))
        O = int(rng.integers(1, 6 * b))
        O = min(O, stride * b - P + 1)
        group, plen = -1, 0
        if sharing and rng.random() < 0.6:
            group = int(rng.integers(0, 3))
            plen = group_len[group]
            if plen > P:
                group, plen = -1, 0
        nb = int(rng.integers(2, N_max + 1)) if budgets else 0
        reqs.append((i, P, O, group, plen, nb))
    return reqs


def _table_list(row):
    return [int(x) for x in row if x >= 0]


@pytest.mark.parametrize("name,policy,sharing,budgets,M,n_total", CASES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_scheduler_matches_oracle(name, policy, sharing, budgets, M, n_total, seed):
    from compressed_paged_kv_zp_gb300.sched import Scheduler
    b, w, N_max, stride, max_running, max_prefill = 4, 2, 5, 24, 12, 40
    rng = np.random.default_rng(1000 * seed + len(name))
    trace = _trace(rng, 30, b, N_max, stride, sharing, budgets)
    cfg = dict(b=b, w=w, N_max=N_max, M=M, policy=policy, prefix_sharing=sharing, max_running=max_running,
               max_prefill_tokens=max_prefill, table_stride=stride)
    ora = OracleScheduler(n_total=n_total, **cfg)
    lib = Scheduler(n_total, b, w, N_max, M, policy=policy, prefix_sharing=sharing, max_running=max_running,
                    max_prefill_tokens=max_prefill, table_stride=stride)
    for r in trace:
        ora.add(*r)
        lib.add(*r)
    budget = {r[0]: (r[5] or N_max) for r in trace}
    outlen = {r[0]: r[2] for r in trace}
    inflight = []  # (due step, id, oracle plan)
    ever_compressed = set()
    n_pre = n_comp = n_blocked = 0
    for step in range(20000):
        still = []
        for due, rid, plan in inflight:
            if due <= step:
                lib.compression_done(rid)
                ora.compression_done(rid, plan)
            else:
                still.append((due, rid, plan))
        inflight = still
        try:
            so = ora.schedule()
        except OracleSchedError:
            with pytest.raises(Exception):
                lib.schedule()
            pytest.fail("deadlock at step %d" % step)
        sl = lib.schedule()
        assert sl["kind"] == so["kind"], step
        assert sl["ids"].tolist() == so["ids"]
        assert sl["lens"].tolist() == so["lens"]
        assert sl["start"].tolist() == so["start"]
        assert sl["slots"].tolist() == so["slots"]
        assert [_table_list(t) for t in sl["tables"]] == so["tables"]
        assert sl["preempted"] == so["preempted"] and sl["blocked"] == so["blocked"]
        assert not set(so["preempted"]) & ever_compressed
        n_pre += len(so["preempted"])
        n_blocked += so["blocked"]
        if so["kind"] == "decode":
            for rid, pos, slot in zip(so["ids"], so["start"], so["slots"]):
                if pos // b + 1 >= budget[rid] and pos % b >= b - w:
                    assert slot >= 0  # window tokens only with a query slot
        fo, po = ora.commit()
        fl, pl = lib.commit()
        assert fl == fo and pl == po
        assert not set(po) & ever_compressed
        n_pre += len(po)
        co = ora.take_compressions()
        cl = lib.take_compressions()
        assert cl["ids"].tolist() == [c["id"] for c in co]
        assert cl["lens"].tolist() == [c["L"] for c in co]
        assert cl["slots"].tolist() == [c["slot"] for c in co]
        assert cl["k"].tolist() == [c["k"] for c in co]
        assert cl["first"].tolist() == [int(c["first"]) for c in co]
        assert [_table_list(t) for t in cl["tables"]] == [c["table"] for c in co]
        for i, c in enumerate(co):
            tg = cl["targets"][i]
            assert _table_list(tg) == c["targets"] and (tg[len(c["targets"]):] == -1).all()
            inflight.append((step + 1 + int(rng.integers(0, 3)), c["id"], c))
            ever_compressed.add(c["id"])
            n_comp += 1
        # invariants
        assert lib.counts() == ora.counts()
        slots = [r.slot for r in ora.running if r.slot >= 0]
        assert len(slots) == len(set(slots)) <= M
        if policy == 0:
            assert len(ora.running) <= M and all(r.slot >= 0 for r in ora.running)
            if not sharing:
                assert n_pre == 0
        for r in ora.running:
            if r.compressed and r.state == 1:
                assert len(r.table) <= budget[r.id]
        held = sum(len(r.table) for r in ora.running)
        fresh = sum(len(set(c[2]["new_table"]) - set(c[2]["table"])) for c in inflight)
        assert int(ora.ref.sum()) == held + fresh  # every reference is accounted for
        if ora.counts()["finished"] == len(trace):
            break
    else:
        pytest.fail("trace did not finish")
    for r in trace:
        info = lib.info(r[0])
        assert info["state"] == 3 and info["generated"] == outlen[r[0]]
    assert lib.counts()["free_blocks"] == n_total and lib.counts()["free_slots"] == M
    assert n_comp > 0
    print(name, seed, "steps", step, "compressions", n_comp, "preemptions", n_pre, "blocked", n_blocked)


def test_bad_arguments_are_refused():
    from compressed_paged_kv_zp_gb300 import ZPError
    from compressed_paged_kv_zp_gb300.sched import Scheduler
    with pytest.raises(ZPError):
        Scheduler(10, 4, 5, 4, 1, table_stride=8)  # w > b
    s = Scheduler(10, 4, 2, 4, 1, table_stride=8)
    s.add(0, 4, 4)
    with pytest.raises(ZPError):
        s.add(0, 4, 4)  # id taken
    with pytest.raises(ZPError):
        s.add(1, 30, 4)  # longer than a block table
    with pytest.raises(ZPError):
        s.add(2, 8, 4, group=1, prefix_len=6)  # prefix not whole blocks
    with pytest.raises(ZPError):
        s.add(3, 8, 4, max_blocks=5)  # budget above N_max
    s.add(4, 8, 4, group=1, prefix_len=4)
    with pytest.raises(ZPError):
        s.add(5, 12, 4, group=1, prefix_len=8)  # a group has one prefix length
    with pytest.raises(ZPError):
        s.compression_done(0)  # not compressing
    s.schedule()
    with pytest.raises(ZPError):
        s.schedule()  # the last step was not committed


def test_deadlock_is_reported():
    from compressed_paged_kv_zp_gb300 import ZPError
    from compressed_paged_kv_zp_gb300.sched import Scheduler
    s = Scheduler(2, 4, 2, 2, 1, policy=0, table_stride=8)
    s.add(0, 12, 2)
    with pytest.raises(ZPError) as e:
        s.schedule()
    assert e.value.status == 4
