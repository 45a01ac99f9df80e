"""The serving loop (native scheduler + kernels) on synthetic traces.

* Constrained and hybrid scheduling, 32q/8kv/128 bf16, b = 16, N_max = 8,
  2 layers: requests that are never preempted (constrained: nobody is; hybrid:
  the requests holding a query slot from their admission) are mirrored by the
  oracle loop from their prefill on -- outputs of every decode step they take
  part in, triggers and keep sets.  Their scores reach the oracle's only if
  each window token was scored into the request's own slot while the batch
  around it changed from step to step.
* Hybrid scheduling with shared prefixes and per-request budgets on a tight
  pool: the run completes with requests blocked and preempted, no device
  error, every block back in the pool and every slot free.
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import TOL_OUT
from tests.oracle_loop import OracleLoop

pytestmark = pytest.mark.gpu

SHAPE = dict(h_q=32, h_kv=8, d=128, b=16)


def _mirror_of(loop, rid, table_row, L):
    blk = torch.from_numpy(table_row[table_row >= 0].astype(np.int64)).to(loop.dev)
    Kb = loop.K.index_select(1, blk).float().cpu().numpy()
    Vb = loop.V.index_select(1, blk).float().cpu().numpy()
    cfg = dict(h_q=loop.h_q, h_kv=loop.h_kv, d=loop.d, b=loop.b, N_max=loop.budget[rid], w=loop.window)
    return OracleLoop.mirror(cfg, [Kb], [Vb], np.array([L]), loop.stride, spare=loop.stride + 4)


@pytest.mark.parametrize("policy", ["constrained", "hybrid"])
def test_served_requests_match_the_oracle(policy):
    from compressed_paged_kv_zp_gb300.serve import ServeLoop, synthetic_trace
    from compressed_paged_kv_zp_gb300.sched import CONSTRAINED, HYBRID
    import compressed_paged_kv_zp_gb300 as zp
    b, N_max, M, layers = 16, 8, 3, 2
    trace = synthetic_trace(18, 71, prompt=(16, 200), output=(60, 330))
    stride = (200 + 330) // b + 2
    loop = ServeLoop(n_total=160, max_blocks=N_max, query_slots=M, table_stride=stride, layers=layers,
                     policy=CONSTRAINED if policy == "constrained" else HYBRID, max_running=12, seed=72, **SHAPE)
    for r in trace:
        loop.add_request(*r)
    watch = {0, 1, 2}  # admitted first, they hold the M slots; slot holders are never preempted without sharing
    mirrors, checked, compared_keeps, swaps = {}, 0, 0, 0
    for _ in range(100000):
        c = loop.sched.counts()
        if c["waiting"] == 0 and c["running"] == 0:
            break
        kind, fin = loop.step()
        ids = [int(x) for x in loop.last_step[1]]
        if kind == "prefill":
            st_tables = {int(i): loop.sched.info(int(i)) for i in ids}
            for i in ids:
                i = int(i)
                if i in watch and i not in mirrors:
                    assert st_tables[i]["slot"] >= 0 and st_tables[i]["preemptions"] == 0
                    row = loop.last_step[3][ids.index(i)]
                    mirrors[i] = _mirror_of(loop, i, row, st_tables[i]["L"])
        elif kind == "decode":
            q, kn, vn = loop.last_step[2]
            for pos, i in enumerate(ids):
                i = int(i)
                if i not in mirrors:
                    continue
                ora = mirrors[i]
                sel = lambda x: x[:, pos:pos + 1].float().cpu().numpy()  # noqa: E731
                out_ref, trig = ora.step(sel(q), sel(kn), sel(vn))
                np.testing.assert_allclose(loop.out[:, pos:pos + 1].float().cpu().numpy(), out_ref, **TOL_OUT["bf16"])
                checked += 1
                info = loop.sched.info(i)
                assert info["preemptions"] == 0
                if i in fin:  # its last token: finished, not compressed
                    assert info["state"] == 3
                    del mirrors[i]
                    continue
                if trig:
                    assert info["state"] == 2  # compressing
                    torch.cuda.synchronize()
                    kids, keep = loop.last_keep
                    swaps += ora.compress(0, keep[:, kids.index(i)].cpu().numpy())
                    compared_keeps += 1
                elif info["state"] == 2:
                    raise AssertionError("device compressed request %d, the oracle did not" % i)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    c = loop.sched.counts()
    assert c["finished"] == len(trace) and c["free_blocks"] == loop.n_total and c["free_slots"] == M
    assert checked > 300 and compared_keeps >= 4
    print(policy, loop.stats, "mirrored steps", checked, "keep sets", compared_keeps, "near-tie swaps", swaps)


def test_tight_pool_hybrid_prefix_sharing_budgets_completes():
    from compressed_paged_kv_zp_gb300.serve import ServeLoop, synthetic_trace
    from compressed_paged_kv_zp_gb300.sched import HYBRID
    import compressed_paged_kv_zp_gb300 as zp
    b, N_max, M, layers = 16, 16, 4, 2
    trace = synthetic_trace(40, 81, prompt=(64, 400), output=(50, 500), prefix_groups=3, prefix_len=48,
                            budgets=(4, 16))
    stride = (400 + 500) // b + 2
    loop = ServeLoop(n_total=200, max_blocks=N_max, query_slots=M, table_stride=stride, layers=layers,
                     policy=HYBRID, prefix_sharing=True, max_running=24, seed=82, **SHAPE)
    for r in trace:
        loop.add_request(*r)
    m = loop.run()
    assert zp.zp_device_status() == (0, 0)
    c = loop.sched.counts()
    assert c["finished"] == len(trace) and c["free_blocks"] == loop.n_total and c["free_slots"] == M
    assert m["compressions"] > 10 and m["preemptions"] > 0 and m["blocked"] > 0
    assert m["tokens"] == sum(r[2] for r in trace) and m["tps"] > 0
    print(m)
