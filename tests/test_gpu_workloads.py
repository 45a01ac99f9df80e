"""The larger decode-with-compression workloads at full size, on the
DecodeLoop driver.

* High concurrency: 32q/8kv/128 bf16, b = 16, 512 sequences starting at
  contexts uniform in [1024, 4096], budget N_max = 128 blocks (2032 tokens
  kept), 2048 decode steps with compression whenever the §4.1 trigger holds.
  Checked: no device error; every sequence compressed; none holds more than
  N_max blocks; the pool accounts for every block; sampled keep sets are
  ascending and complete; two sequences (the longest, and the shortest that
  starts above the budget) mirrored by the oracle loop for the first 256
  steps: outputs every step (after a compression they read the moved rows),
  triggers and keep sets.
* Prefix-shared, 36 layers: 32q/8kv/128 bf16, 256 sequences sharing a
  1024-token prefix (64 blocks), private tails uniform in [0, 8192], budget
  N_max = 64 blocks, compression asynchronous on the side stream while the
  others decode, 8 layers per compression call (App. C.1's layer stride).  A prefix cache holds one more reference to the prefix, so
  every compaction must go to fresh target blocks (§4.4).  Checked: the
  prefix blocks are never written; after all sequences compressed, only the
  prefix cache holds them; the sequences' blocks are disjoint and at most
  N_max each; the pool accounts for every block; two sequences mirrored by
  the oracle loop on the first and last layer over all steps they decode.
  The ~194 GB of K and V run at once when the device has the room, else in
  waves of 128 or 64 sequences (printed).
The cache contents and per-step inputs are drawn on the device from seeded
generators; the oracle loops start from a copy of the mirrored sequences'
blocks taken before any kernel ran and then keep their own state.
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import TOL_OUT
from tests.oracle_loop import OracleLoop

pytestmark = pytest.mark.gpu


def _dev_normal(shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)


def _check_pool(loop, extra=()):
    held = {}
    for x in list(loop.table[loop.table >= 0].ravel()) + list(extra):
        held[int(x)] = held.get(int(x), 0) + 1
    for blk, r in held.items():
        assert loop.pool.refcount(blk) == r, (blk, r)
    assert loop.pool.num_free + len(held) == loop.n_total


def _mirror(loop, seqs, layers, N_max, w):
    """An oracle loop over `seqs` on `layers`, from the blocks they hold now."""
    Kb, Vb = [], []
    lidx = torch.tensor(layers, device=loop.K.device)
    for s in seqs:
        blk = torch.from_numpy(loop.table[s][loop.table[s] >= 0].astype(np.int64)).to(loop.K.device)
        Kb.append(loop.K.index_select(0, lidx).index_select(1, blk).float().cpu().numpy())
        Vb.append(loop.V.index_select(0, lidx).index_select(1, blk).float().cpu().numpy())
    cfg = dict(h_q=loop.h_q, h_kv=loop.h_kv, d=loop.d, b=loop.b, N_max=N_max, w=w)
    return OracleLoop.mirror(cfg, Kb, Vb, loop.lens[seqs], loop.stride, spare=loop.stride + 4)


def _mirror_step(ora, loop, seqs, layers, q, kn, vn, trig):
    """One step of the oracle loop; compares outputs, triggers and (at a
    compression) keep sets with the device.  Returns reported near-ties."""
    li = torch.tensor(layers, device=q.device)
    si = torch.from_numpy(np.asarray(seqs, dtype=np.int64)).to(q.device)
    pick = lambda x: x.index_select(0, li).index_select(1, si).float().cpu().numpy()
    out_ref, trig_ref = ora.step(pick(q), pick(kn), pick(vn))
    np.testing.assert_allclose(pick(loop.out), out_ref, **TOL_OUT["bf16"])
    assert [seqs[i] for i in trig_ref] == [s for s in seqs if s in set(trig)]
    swaps = 0
    if trig_ref:
        torch.cuda.synchronize()  # the keep sets are written on the side stream
        gseqs, keep = loop.last_keep
        keep = keep.index_select(0, li).cpu().numpy()
        pos = {int(x): i for i, x in enumerate(gseqs)}
        for i in trig_ref:
            swaps += ora.compress(i, keep[:, pos[seqs[i]]])
    return swaps


def test_high_concurrency_512_sequences_2048_steps():
    from compressed_paged_kv_zp_gb300.engine import DecodeLoop
    B, h_q, h_kv, d, b, N_max, steps = 512, 32, 8, 128, 16, 128, 2048
    g = torch.Generator().manual_seed(1003)
    lens0 = torch.randint(1024, 4097, (B,), generator=g).numpy().astype(np.int32)
    stride = 4096 // b + 2
    n_total = int(np.maximum((lens0 + b - 1) // b + 1, N_max).sum()) + 64
    loop = DecodeLoop(h_q, h_kv, d, b, n_total, N_max, stride, layers=1, dtype=torch.bfloat16, window=b)
    loop.add_sequences(lens0)
    loop.K.copy_(_dev_normal(loop.K.shape, 11))
    loop.V.copy_(_dev_normal(loop.V.shape, 12))
    above = np.nonzero(lens0 > N_max * b)[0]
    mseqs = [int(above[np.argmin(lens0[above])]), int(np.argmax(lens0))]
    ora = _mirror(loop, mseqs, [0], N_max, b)
    compressed = np.zeros(B, dtype=bool)
    swaps = 0
    for step in range(steps):
        q = _dev_normal((1, B, h_q, d), 100000 + step)
        kn = _dev_normal((1, B, h_kv, d), 200000 + step)
        vn = _dev_normal((1, B, h_kv, d), 300000 + step)
        trig = loop.step(q, kn, vn)
        if step < 256:
            swaps += _mirror_step(ora, loop, mseqs, [0], q, kn, vn, trig)
        if trig:
            compressed[trig] = True
            if step % 97 == 0:
                seqs, keep = loop.last_keep
                kp = keep[0].cpu().numpy()  # [n][h_kv][k]
                assert np.all(np.diff(kp, axis=-1) > 0) and np.all(kp[..., 0] >= 0)
    assert not ora.first.any()  # both mirrored sequences compressed
    loop.drain()
    torch.cuda.synchronize()
    import compressed_paged_kv_zp_gb300 as zp
    assert zp.zp_device_status() == (0, 0)
    assert compressed.all()
    assert (loop.table >= 0).sum(axis=1).max() <= N_max
    _check_pool(loop)
    print("compressions:", loop.compressions, "reported near-tie swaps:", swaps)


def test_per_request_budgets_in_the_loop():
    """Per-request block budgets N_i uniform in [4, 128] (N_max = 128) on 48
    sequences at contexts uniform in [1024, 4096], 600 steps, compression on
    the side stream: every request compresses at its own N_i to (N_i - 1) b
    tokens; two requests with different budgets mirrored by the oracle loop
    at their own N_i over all steps (outputs, triggers, keep sets)."""
    from compressed_paged_kv_zp_gb300.engine import DecodeLoop
    B, h_q, h_kv, d, b, N_max, steps = 48, 32, 8, 128, 16, 128, 600
    g = torch.Generator().manual_seed(1007)
    lens0 = torch.randint(1024, 4097, (B,), generator=g).numpy().astype(np.int32)
    N_i = torch.randint(4, N_max + 1, (B,), generator=g).numpy().astype(np.int32)
    N_i[0], N_i[1] = 4, 37
    stride = 4096 // b + 2
    n_total = int(np.maximum((lens0 + b - 1) // b + 1, N_i).sum()) + 64
    loop = DecodeLoop(h_q, h_kv, d, b, n_total, N_max, stride, layers=1, dtype=torch.bfloat16, window=b,
                      async_compress=True)
    loop.add_sequences(lens0, max_blocks=N_i)
    loop.K.copy_(_dev_normal(loop.K.shape, 31))
    loop.V.copy_(_dev_normal(loop.V.shape, 32))
    mseqs = [0, 1]
    oras = [_mirror(loop, [s], [0], int(N_i[s]), b) for s in mseqs]
    count = np.zeros(B, dtype=np.int64)
    swaps, checked = 0, 0
    for step in range(steps):
        q = _dev_normal((1, B, h_q, d), 700000 + step)
        kn = _dev_normal((1, B, h_kv, d), 800000 + step)
        vn = _dev_normal((1, B, h_kv, d), 900000 + step)
        trig = loop.step(q, kn, vn)
        if trig:
            again = [x for x in trig if count[x] > 0]  # a compressed request grows back to N_i blocks
            assert (loop.lens[again] == N_i[again] * b).all()
            plan = loop.pending[-1][2]
            for i, s in enumerate(trig):  # targets and new table padded past the request's own budget
                assert (plan["targets"][i, N_i[s] - 1:] == -1).all() and (plan["targets"][i, :N_i[s] - 1] >= 0).all()
                assert (plan["new_tables"][i, N_i[s]:] == -1).all()
        count[trig] += 1
        for s, ora in zip(mseqs, oras):
            if loop.active[s] or s in trig:
                swaps += _mirror_step(ora, loop, [s], [0], q, kn, vn, trig)
                checked += 1
    loop.drain()
    torch.cuda.synchronize()
    import compressed_paged_kv_zp_gb300 as zp
    assert zp.zp_device_status() == (0, 0)
    due = lens0 + steps >= N_i * b + b
    assert (count[due] > 0).all()
    assert count[0] >= 20  # N_0 = 4 blocks: a compression every 16 decoded steps
    held = (loop.table >= 0).sum(axis=1)
    assert (held <= N_i).all()
    _check_pool(loop)
    assert not any(o.first.any() for o in oras)
    print("compressions:", loop.compressions, "mirrored steps:", checked, "reported near-tie swaps:", swaps)


def _prefix_shared_wave(B, lens0, seed, steps, mirror):
    """One DecodeLoop over B sequences sharing a 1024-token prefix (64 blocks,
    plus the prefix cache's own reference) on 36 layers, N_max = 64, steps
    decode steps with asynchronous compression (8 layers per call); the
    longest and the shortest sequence mirrored by the oracle loop on the first
    and last layer when `mirror`."""
    from compressed_paged_kv_zp_gb300.engine import DecodeLoop
    h_q, h_kv, d, b, N_max, layers = 32, 8, 128, 16, 64, 36
    g = torch.Generator().manual_seed(seed)
    P = 1024 // b
    stride = (int(lens0.max()) + steps + b - 1) // b + 2
    own = (lens0 + b - 1) // b - P
    n_total = P + int(own.sum()) + B * (N_max + 2) + 64
    table = np.full((B, stride), -1, dtype=np.int32)
    perm = torch.randperm(n_total, generator=g).numpy().astype(np.int32)
    table[:, :P] = perm[:P]
    cur = P
    for s in range(B):
        table[s, P:P + own[s]] = perm[cur:cur + own[s]]
        cur += own[s]
    loop = DecodeLoop(h_q, h_kv, d, b, n_total, N_max, stride, layers=layers, dtype=torch.bfloat16, window=b,
                      async_compress=True, layer_stride=8)  # 8 layers per compression call
    loop.add_sequences(lens0, tables=table)
    prefix = table[0, :P].copy()
    loop.pool.incref(prefix.tolist())  # the prefix cache's own reference
    for l in range(layers):  # layer by layer: no fp32 copy of the whole cache
        loop.K[l].copy_(_dev_normal(loop.K[l].shape, seed * 100 + 2 * l))
        loop.V[l].copy_(_dev_normal(loop.V[l].shape, seed * 100 + 2 * l + 1))
    pidx = torch.from_numpy(prefix.astype(np.int64)).cuda()
    K_prefix = loop.K.index_select(1, pidx).clone()
    V_prefix = loop.V.index_select(1, pidx).clone()
    assert all(loop.pool.refcount(int(x)) == B + 1 for x in prefix)
    mseqs = [int(np.argmax(lens0)), int(np.argmin(lens0))] if mirror else []
    mlayers = [0, layers - 1]
    oras = [_mirror(loop, [s], mlayers, N_max, b) for s in mseqs]
    seen = np.zeros(B, dtype=bool)
    checked, swaps = 0, 0
    for step in range(steps):
        q = _dev_normal((layers, B, h_q, d), seed * 1000 + 3 * step)
        kn = _dev_normal((layers, B, h_kv, d), seed * 1000 + 3 * step + 1)
        vn = _dev_normal((layers, B, h_kv, d), seed * 1000 + 3 * step + 2)
        trig = loop.step(q, kn, vn)
        seen[trig] = True
        if trig:
            plan = loop.pending[-1][2]
            assert not set(plan["targets"].ravel().tolist()) & set(prefix.tolist())
        for s, ora in zip(mseqs, oras):
            if loop.active[s] or s in trig:  # decoded in this step
                swaps += _mirror_step(ora, loop, [s], mlayers, q, kn, vn, trig)
                checked += 1
    loop.drain()
    torch.cuda.synchronize()
    import compressed_paged_kv_zp_gb300 as zp
    assert zp.zp_device_status() == (0, 0)
    assert seen.all()
    assert torch.equal(loop.K.index_select(1, pidx), K_prefix)
    assert torch.equal(loop.V.index_select(1, pidx), V_prefix)
    assert all(loop.pool.refcount(int(x)) == 1 for x in prefix)
    assert not set(loop.table[loop.table >= 0].tolist()) & set(prefix.tolist())
    held = [loop.table[s][loop.table[s] >= 0] for s in range(B)]
    assert max(len(h) for h in held) <= N_max
    allb = np.concatenate(held)
    assert len(np.unique(allb)) == len(allb)
    _check_pool(loop, extra=prefix.tolist())
    assert not any(o.first.any() for o in oras)
    comps = loop.compressions
    del loop, K_prefix, V_prefix
    torch.cuda.empty_cache()
    return comps, checked, swaps


def test_prefix_shared_36_layers_async():
    """The prefix-shared workload at its stated size: 256 sequences, a shared
    1024-token prefix plus private tails uniform in [0, 8192], 36 layers of
    32q/8kv/128 bf16, N_max = 64 (1008 kept), 40 steps (every sequence
    compresses at least twice).  K and V of all 256 sequences take ~194 GB;
    when the device has less free memory the batch runs in waves of 128 or 64
    sequences (each wave its own pool and its own copy of the prefix), and the
    test says which it ran."""
    B, steps = 256, 40
    g = torch.Generator().manual_seed(1005)
    lens0 = (1024 + torch.randint(0, 8193, (B,), generator=g).numpy()).astype(np.int32)
    blocks = int(((lens0 + 15) // 16).sum()) + B * 66
    need = blocks * 36 * 16 * 8 * 128 * 2 * 2 * 1.06 + 12e9  # K, V, scores, scratch
    torch.cuda.empty_cache()
    free = torch.cuda.mem_get_info()[0]
    waves = 1 if need <= free else (2 if need / 2 <= free else 4)
    per = B // waves
    tot_c = tot_chk = tot_sw = 0
    for w in range(waves):
        c, chk, sw = _prefix_shared_wave(per, lens0[w * per:(w + 1) * per], 1005 + w, steps, mirror=(w == 0))
        tot_c += c
        tot_chk += chk
        tot_sw += sw
    assert tot_chk > 40 and tot_c >= 3 * B // 2
    print("waves:", waves, "compressions:", tot_c, "mirrored steps:", tot_chk, "reported near-tie swaps:", tot_sw)
