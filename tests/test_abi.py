"""C ABI checks and host logic that need no GPU.

* libzp.so loads and exports every function include/*.h declares;
* the trigger and the host block pool / planner agree with the oracle's
  reading of [Zipage §4.1, §4.4] on random tables with shared prefixes;
* calls with invalid arguments fail with the documented status before any
  device work.
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def zp():
    import compressed_paged_kv_zp_gb300 as m
    return m


def _declared():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, h)).read() for h in sorted(os.listdir(inc)) if h.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(zp_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_binding_exports(zp):
    assert sorted(zp.EXPORTS) == _declared()


def test_every_declared_symbol_is_exported(zp):
    for name in _declared():
        assert hasattr(zp.lib, name), name
        assert ctypes.cast(getattr(zp.lib, name), ctypes.c_void_p).value


def test_status_strings(zp):
    for code, name in zp.STATUS.items():
        assert zp.lib.zp_status_string(code).decode() == name
    assert zp.lib.zp_version() >= 1


def test_trigger_matches_oracle(zp, orc):
    for b in (4, 16):
        for N_max in (2, 4, 8):
            for L in range(0, 12 * b):
                assert zp.zp_needs_compression(L, b, N_max) == orc.needs_compression(L, b, N_max)


def test_batched_trigger_matches_oracle(zp, orc):
    """The batched trigger returns exactly the active sequences whose
    per-sequence trigger holds in the oracle, with uniform and per-request
    budgets."""
    rng = np.random.default_rng(5)
    for b in (4, 16):
        lens = rng.integers(0, 40 * b, size=300).astype(np.int32)
        lens[::7] = (lens[::7] // b) * b  # many block-aligned lengths
        active = rng.random(300) < 0.8
        per = rng.integers(2, 33, size=300).astype(np.int32)
        for N_max, budgets in ((8, None), (32, per)):
            got = zp.zp_needs_compression_batch(lens, b, N_max, active=active, max_blocks_seq=budgets)
            want = [i for i in range(300) if active[i] and orc.needs_compression(
                int(lens[i]), b, int(budgets[i]) if budgets is not None else N_max)]
            assert got.tolist() == want
    assert zp.zp_needs_compression_batch(np.zeros(0, np.int32), 16, 8).tolist() == []


@pytest.mark.parametrize("seed", range(12))
def test_planner_matches_oracle(zp, orc, seed):
    rng = np.random.default_rng(seed)
    n_total = 64
    pool = zp.Pool(n_total)
    N_max = int(rng.integers(2, 7))
    N = int(rng.integers(N_max, N_max + 5))
    n_prefix = int(rng.integers(0, N + 1))
    prefix = pool.alloc(n_prefix)
    sharers = int(rng.integers(1, 4))
    for _ in range(sharers - 1):
        pool.incref(prefix)
    own = pool.alloc(N - n_prefix)
    table = prefix + own
    ref = np.array([pool.refcount(i) for i in range(n_total)], dtype=np.int32)
    free_before = pool.num_free
    # the oracle takes fresh blocks in the order the pool hands them out
    fresh = sorted(set(range(n_total)) - {i for i in range(n_total) if ref[i] > 0})
    plan_o = orc.plan_targets(np.array(table, dtype=np.int32), N_max, ref,
                              np.array(fresh, dtype=np.int32))
    plan = pool.plan_compaction(table, N_max)
    assert plan["targets"] == list(plan_o["targets"])
    assert plan["new_table"] == list(plan_o["new_table"])
    assert sorted(plan["dropped"]) == sorted(list(plan_o["released"]) + list(plan_o["dropped_shared"]))
    assert plan["n_fresh"] == plan_o["fresh_used"] == pool.n_total - pool.num_free - (n_total - free_before)
    # release what the sequence no longer holds: own blocks return to the pool,
    # shared ones lose one reference
    pool.release(plan["dropped"])
    for blk in plan_o["released"]:
        assert pool.refcount(int(blk)) == 0
    for blk in plan_o["dropped_shared"]:
        assert pool.refcount(int(blk)) == ref[blk] - 1
    held = sum(1 for i in range(n_total) if pool.refcount(i) > 0)
    assert held + pool.num_free == n_total  # conservation


def test_pool_errors(zp):
    pool = zp.Pool(4)
    with pytest.raises(zp.ZPError) as e:
        pool.alloc(5)
    assert e.value.status == 4
    ids = pool.alloc(2)
    with pytest.raises(zp.ZPError):
        pool.release([ids[0], ids[0]])  # over-release
    pool.release(ids)
    assert pool.num_free == 4
    with pytest.raises(zp.ZPError):
        pool.plan_compaction([0, 1], 3)  # fewer blocks than the budget


def test_invalid_arguments_rejected_without_device(zp):
    desc = zp.cache_desc(8, 3, 64, 16, 10, 0)  # h_q % h_kv != 0
    rc = zp.lib.zp_append_kv(ctypes.byref(desc), None, None, None, None, None, 1, None, 1, None)
    assert rc == 2
    desc = zp.cache_desc(8, 2, 64, 16, 10, 9)  # bad dtype
    rc = zp.lib.zp_select_topk(None, 2, 4, None, 1, 2, None, None, None, None)
    assert rc == 1
    rc = zp.lib.zp_compact_pages(ctypes.byref(desc), None, None, 0, 1, None, 0, None, None, 1, None, 1,
                                 None, None, 4, None, 1, None)
    assert rc == 3
    # global_F without the score rows it is written from
    desc = zp.cache_desc(8, 2, 64, 16, 10, 0)
    one = ctypes.c_void_p(16)  # never dereferenced: the call fails its argument checks first
    rc = zp.lib.zp_compact_pages(ctypes.byref(desc), one, one, 0, 1, one, 0, None, one, 1, one, 1,
                                 one, one, 4, None, 1, None)
    assert rc == 1
    # score_tokens without attention-score rows
    rc = zp.lib.zp_score_tokens(ctypes.byref(desc), ctypes.byref(zp.score_params()), one, one, 1, one, one, 1,
                                None, one, one, 4, one, 1 << 30, None)
    assert rc == 1


def test_batch_planner_matches_single_calls(zp):
    import numpy as np
    rng = np.random.default_rng(11)
    pools = [zp.Pool(400), zp.Pool(400)]
    n, stride, N_max = 6, 12, 5
    tables = np.full((n, stride), -1, np.int32)
    nb = rng.integers(N_max, stride + 1, size=n).astype(np.int32)
    for pool in pools:  # identical histories: shared prefix of 3 blocks for all
        prefix = pool.alloc(3)
        for _ in range(n - 1):
            pool.incref(prefix)
        for i in range(n):
            tables[i, :3] = prefix
            tables[i, 3:nb[i]] = pool.alloc(int(nb[i]) - 3)
    singles = [pools[0].plan_compaction(tables[i, :nb[i]].tolist(), N_max) for i in range(n)]
    batch = pools[1].plan_compaction_batch(tables, nb, N_max)
    for i, sp in enumerate(singles):
        assert list(batch["targets"][i]) == sp["targets"]
        assert list(batch["new_tables"][i]) == sp["new_table"]
        assert list(batch["dropped"][i, :batch["n_dropped"][i]]) == sp["dropped"]
        assert batch["n_fresh"][i] == sp["n_fresh"]
    assert pools[0].num_free == pools[1].num_free


def test_batch_planner_per_request_budgets(zp):
    """Per-request block budgets: each row equals a single plan with that
    sequence's own budget, padded with -1 up to the batch's largest budget;
    a budget outside [2, max_blocks] is refused."""
    import numpy as np
    rng = np.random.default_rng(12)
    pools = [zp.Pool(500), zp.Pool(500)]
    n, stride, N_max = 7, 14, 8
    mb = rng.integers(2, N_max + 1, size=n).astype(np.int32)
    mb[0], mb[1] = 2, N_max
    tables = np.full((n, stride), -1, np.int32)
    nb = np.array([rng.integers(int(m), stride + 1) for m in mb], np.int32)
    for pool in pools:
        prefix = pool.alloc(2)
        for _ in range(n - 1):
            pool.incref(prefix)
        for i in range(n):
            tables[i, :2] = prefix
            tables[i, 2:nb[i]] = pool.alloc(int(nb[i]) - 2)
    singles = [pools[0].plan_compaction(tables[i, :nb[i]].tolist(), int(mb[i])) for i in range(n)]
    batch = pools[1].plan_compaction_batch(tables, nb, N_max, max_blocks_seq=mb)
    for i, sp in enumerate(singles):
        m = int(mb[i])
        assert list(batch["targets"][i, :m - 1]) == sp["targets"]
        assert (batch["targets"][i, m - 1:] == -1).all()
        assert list(batch["new_tables"][i, :m]) == sp["new_table"]
        assert (batch["new_tables"][i, m:] == -1).all()
        assert list(batch["dropped"][i, :batch["n_dropped"][i]]) == sp["dropped"]
        assert batch["n_fresh"][i] == sp["n_fresh"]
    assert pools[0].num_free == pools[1].num_free
    with pytest.raises(zp.ZPError):
        pools[1].plan_compaction_batch(tables[:1], nb[:1], N_max, max_blocks_seq=np.array([N_max + 1], np.int32))
    with pytest.raises(zp.ZPError):
        pools[1].plan_compaction_batch(tables[:1], nb[:1], N_max, max_blocks_seq=np.array([1], np.int32))


def test_capacity_plan_brute_force(zp):
    """eq. (1)/(2): M is the largest concurrency any block count allows; the
    returned N_total is feasible with it and equals the linear program's
    optimum (floored) -- checked against enumeration on small budgets."""
    import random
    from fractions import Fraction
    rng = random.Random(5)
    for _ in range(200):
        A = rng.randint(50, 1200)
        m = rng.randint(1, 40)
        q = rng.randint(0, 60)
        N = rng.randint(1, 9)
        num, den = rng.choice([(0, 1), (1, 16), (1, 256), (3, 7)])
        f = Fraction(num, den)
        best = 0
        for Nt in range(1, A // m + 2):
            for M in range(1, Nt // N + 1):
                if (1 + f) * m * Nt + M * q <= A:
                    best = max(best, M)
        if best == 0:
            with pytest.raises(zp.ZPError):
                zp.zp_plan_capacity(A, m, q, N, (num, den))
            continue
        M, Nt = zp.zp_plan_capacity(A, m, q, N, (num, den))
        assert M == best
        assert (1 + f) * m * Nt + M * q <= A and M <= Fraction(Nt, N)
        assert Nt == int(Fraction(A) / ((1 + f) * m + Fraction(q, N)))


def test_capacity_plan_closed_forms(zp):
    # no per-request memory: every byte goes to blocks
    assert zp.zp_plan_capacity(1000, 10, 0, 4) == (25, 100)
    # the global score cache at the paper's ratio 1/(2d), d = 128: blocks cost 257/256
    M, N = zp.zp_plan_capacity(257 * 1000, 256, 0, 8, (1, 256))
    assert (M, N) == (125, 1000)
