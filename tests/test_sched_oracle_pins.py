"""Pins of the scheduler oracle (oracle/sched.py) to what the pages state,
on small hand-worked scenarios:

* §4.3 constrained scheduling: concurrency never exceeds M; a request that
  finds no free block waits and nobody is preempted;
* §4.3 hybrid scheduling: concurrency is no longer bounded by M; a request
  without a query slot stops at the observation window of its N_max-th block
  and resumes when a slot is freed; the preemption victim is the last running
  request without a slot;
* §4.1 / Fig. 1: a request compresses after the decode step that fills its
  N_max-th block, keeps (N_max - 1) b tokens in its first N_max - 1 blocks,
  reserves the N_max-th and releases the rest;
* §4.4: with prefix sharing the targets of a request holding shared blocks
  are new blocks, the shared prefix survives, and the request preempted when
  no block is left is the last uncompressed one, slot or not;
* token accounting: a request yields O tokens, one at prefill and one per
  decode step.
"""
import pytest

from oracle.sched import CONSTRAINED, COMPRESSING, FINISHED, HYBRID, OracleSchedError, Scheduler


def _run_until_done(s, limit=10000, on_step=None):
    steps = []
    for _ in range(limit):
        for c in s.take_compressions():
            s.compression_done(c["id"], c)
        st = s.schedule()
        fin, pre = s.commit()
        steps.append((st, fin, pre))
        if on_step:
            on_step(st, fin, pre)
        if all(r.state == FINISHED for r in s.reqs.values()):
            return steps
    raise AssertionError("did not finish")


def test_constrained_concurrency_is_at_most_M():
    s = Scheduler(n_total=100, b=4, w=2, N_max=8, M=2, policy=CONSTRAINED, prefix_sharing=False, max_running=16,
                  max_prefill_tokens=1000, table_stride=16)
    for i in range(3):
        s.add(i, 3, 5)
    st = s.schedule()
    assert st["kind"] == "prefill" and st["ids"] == [0, 1] and st["slots"] == [0, 1]
    s.commit()
    seen_max = 0

    def check(st, fin, pre):
        nonlocal seen_max
        seen_max = max(seen_max, len(s.running))
        assert not pre
    _run_until_done(s, on_step=check)
    assert seen_max == 2


def test_constrained_blocks_instead_of_preempting():
    # 4 blocks of 4 tokens; two requests of 8 prompt tokens each hold 2 blocks,
    # both need a third block at their first decode: one waits, nobody is preempted
    s = Scheduler(n_total=5, b=4, w=2, N_max=3, M=2, policy=CONSTRAINED, prefix_sharing=False, max_running=4,
                  max_prefill_tokens=100, table_stride=8)
    s.add(0, 8, 3)
    s.add(1, 8, 3)
    st = s.schedule()
    assert st["kind"] == "prefill" and st["ids"] == [0, 1]
    s.commit()
    st = s.schedule()
    assert st["kind"] == "decode" and st["ids"] == [0] and st["blocked"] == 1 and not st["preempted"]


def test_hybrid_concurrency_exceeds_M():
    s = Scheduler(n_total=100, b=4, w=2, N_max=8, M=1, policy=HYBRID, prefix_sharing=False, max_running=16,
                  max_prefill_tokens=1000, table_stride=16)
    for i in range(4):
        s.add(i, 3, 6)
    st = s.schedule()
    assert st["kind"] == "prefill" and st["ids"] == [0, 1, 2, 3] and st["slots"] == [0, -1, -1, -1]
    s.commit()
    st = s.schedule()
    assert st["kind"] == "decode" and st["ids"] == [0, 1, 2, 3]


def test_hybrid_slotless_request_stops_at_the_window_and_resumes():
    # b = 4, w = 2, N_max = 2: window positions of block 1 are 6 and 7.
    s = Scheduler(n_total=100, b=4, w=2, N_max=2, M=1, policy=HYBRID, prefix_sharing=False, max_running=4,
                  max_prefill_tokens=100, table_stride=8)
    s.add(0, 2, 5)   # holds the slot, finishes after 4 decode steps
    s.add(1, 2, 20)  # no slot
    s.schedule()
    s.commit()
    positions = []
    for _ in range(4):
        st = s.schedule()
        i = st["ids"].index(1)
        positions.append(st["start"][i])
        s.commit()
    assert positions == [2, 3, 4, 5]  # the new token's position
    assert s.reqs[0].state == FINISHED  # 1 token at prefill + 4 decode steps
    assert s.reqs[1].slot == 0  # the freed slot went to it at commit
    st = s.schedule()
    assert st["ids"] == [1] and st["start"] == [6]


def test_hybrid_slotless_request_blocked_while_slot_is_held():
    s = Scheduler(n_total=100, b=4, w=2, N_max=2, M=1, policy=HYBRID, prefix_sharing=False, max_running=4,
                  max_prefill_tokens=100, table_stride=16)
    s.add(0, 2, 30)
    s.add(1, 2, 30)
    s.schedule()
    s.commit()
    for _ in range(4):
        s.schedule()
        s.commit()
    st = s.schedule()
    assert 1 not in st["ids"] and st["blocked"] == 1  # request 1 waits at position 6


def test_hybrid_preempts_the_last_request_without_a_slot():
    # 4 blocks: three requests of 4 prompt tokens (1 block each) with M = 1;
    # request 0 holds the slot.  Fill the pool, then the slot holder needs a
    # block: the victim is request 2 (the last without a slot), not 0 or 1.
    s = Scheduler(n_total=4, b=4, w=1, N_max=8, M=1, policy=HYBRID, prefix_sharing=False, max_running=4,
                  max_prefill_tokens=100, table_stride=8)
    s.add(0, 4, 20)
    s.add(1, 4, 20)
    s.add(2, 4, 20)
    st = s.schedule()
    assert st["ids"] == [0, 1, 2]
    s.commit()
    st = s.schedule()  # every request needs a second block, one is free
    assert st["ids"] == [0, 1] and st["preempted"] == [2]
    assert s.reqs[2].preemptions == 1 and s.waiting[0].id == 2


def test_trigger_and_targets_follow_fig1():
    # N_max = 4, b = 4: the request holds 4 blocks once its 16th token is cached
    s = Scheduler(n_total=20, b=4, w=2, N_max=4, M=1, policy=HYBRID, prefix_sharing=False, max_running=4,
                  max_prefill_tokens=100, table_stride=8)
    s.add(0, 15, 10)
    st = s.schedule()
    assert st["tables"] == [[0, 1, 2, 3]]
    s.commit()
    st = s.schedule()
    assert st["kind"] == "decode" and st["lens"] == [16]
    s.commit()
    comp = s.take_compressions()
    assert len(comp) == 1
    c = comp[0]
    assert c["L"] == 16 and c["k"] == 12 and c["targets"] == [0, 1, 2] and c["new_table"] == [0, 1, 2, 3]
    assert s.reqs[0].state == COMPRESSING
    assert s.schedule()["kind"] == "idle"  # it sits out until its compression completes
    s.commit()
    s.compression_done(0, c)
    assert s.reqs[0].L == 12 and len(s.reqs[0].table) == 4
    st = s.schedule()
    assert st["start"] == [12] and st["tables"] == [[0, 1, 2, 3]]  # decodes into the reserved block


def test_long_prompt_releases_blocks_at_first_compression():
    s = Scheduler(n_total=40, b=4, w=2, N_max=3, M=1, policy=HYBRID, prefix_sharing=False, max_running=4,
                  max_prefill_tokens=100, table_stride=16)
    s.add(0, 31, 5)  # 8 blocks at prefill
    s.schedule()
    s.commit()
    assert s.counts()["free_blocks"] == 32
    s.schedule()  # caches token 31: the last block is full, N = 8 >= 3
    s.commit()
    (c,) = s.take_compressions()
    assert c["targets"] == [0, 1] and c["new_table"] == [0, 1, 2] and sorted(c["dropped"]) == [3, 4, 5, 6, 7]
    s.compression_done(0, c)
    assert s.counts()["free_blocks"] == 37


def test_prefix_sharing_targets_are_new_blocks_and_prefix_survives():
    s = Scheduler(n_total=40, b=4, w=2, N_max=3, M=2, policy=HYBRID, prefix_sharing=True, max_running=4,
                  max_prefill_tokens=100, table_stride=16)
    s.add(0, 11, 20, group=7, prefix_len=8)
    s.add(1, 11, 20, group=7, prefix_len=8)
    st = s.schedule()
    assert st["tables"] == [[0, 1, 2], [0, 1, 3]] and st["start"] == [0, 8]
    s.commit()
    s.schedule()  # both cache token 11: 3 blocks, last full -> compress
    s.commit()
    comps = s.take_compressions()
    assert [c["id"] for c in comps] == [0, 1]
    assert comps[0]["targets"] == [4, 5]  # blocks 0 and 1 are shared: new targets
    assert comps[0]["new_table"] == [4, 5, 2]
    assert comps[1]["targets"] == [6, 7]  # still shared by request 0's table until its compaction completes
    for c in comps:
        s.compression_done(c["id"], c)
    assert s.ref[0] == 0 and s.ref[1] == 0  # nobody holds the prefix any more


def test_prefix_sharing_preempts_the_last_uncompressed_request_with_a_slot():
    # constrained + sharing: 5 blocks; two requests share a 1-block prefix and
    # hold 2 blocks more each (5 used); request 0 needs a block: request 1 (the
    # last uncompressed, holding a slot) is preempted.
    s = Scheduler(n_total=5, b=4, w=1, N_max=8, M=2, policy=CONSTRAINED, prefix_sharing=True, max_running=4,
                  max_prefill_tokens=100, table_stride=16)
    s.add(0, 12, 30, group=1, prefix_len=4)
    s.add(1, 12, 30, group=1, prefix_len=4)
    st = s.schedule()
    assert st["slots"] == [0, 1] and s.counts()["free_blocks"] == 0
    s.commit()
    st = s.schedule()
    assert st["preempted"] == [1] and st["ids"] == [0]


def test_token_accounting():
    s = Scheduler(n_total=100, b=4, w=2, N_max=8, M=4, policy=HYBRID, prefix_sharing=False, max_running=8,
                  max_prefill_tokens=100, table_stride=16)
    outs = [1, 2, 7]
    for i, o in enumerate(outs):
        s.add(i, 5, o)
    decoded = {i: 0 for i in range(3)}

    def count(st, fin, pre):
        if st["kind"] == "decode":
            for i in st["ids"]:
                decoded[i] += 1
    _run_until_done(s, on_step=count)
    assert [decoded[i] for i in range(3)] == [o - 1 for o in outs]
    assert all(s.reqs[i].generated == outs[i] for i in range(3))


def test_deadlock_is_reported():
    s = Scheduler(n_total=2, b=4, w=2, N_max=2, M=1, policy=CONSTRAINED, prefix_sharing=False, max_running=4,
                  max_prefill_tokens=100, table_stride=16)
    s.add(0, 12, 2)  # needs 3 blocks at prefill, the pool has 2
    with pytest.raises(OracleSchedError):
        s.schedule()
