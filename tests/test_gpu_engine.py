"""Multi-step decode with compression: the DecodeLoop driver against an oracle
loop, step by step (the high-concurrency workload, scaled down).

Every step both sides grow the block tables (lowest free block first), append
the new token, run decode with the window-score accumulation and apply the
§4.1 trigger; triggered sequences are scored, ranked and compacted into the
§4.4 target blocks, their tables swapped, and the blocks they dropped
released.  Checked every step: attention outputs (tolerance), block tables,
lengths and the free pool (exact); at every compression: keep sets (exact up
to reported near-ties, after which the oracle adopts the GPU's choice so both
states stay identical), the moved K/V rows (bit-exact) and F.  The loop runs
with the lightning row sums formed by the decode (the default) and, in one
case, formed by the compression itself.
"""
import numpy as np
import pytest
import torch

import zp_inputs
from tests.gpu_util import TOL_OUT
from tests.oracle_loop import OracleLoop

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layers,async_compress,decode_rho", [(1, False, True), (2, False, True), (2, True, True),
                                                               (2, True, False)])
def test_decode_loop_matches_oracle_loop(layers, async_compress, decode_rho):
    from compressed_paged_kv_zp_gb300.engine import DecodeLoop
    cfg = dict(h_q=16, h_kv=4, d=64, b=16, N_max=4, w=16, layers=layers, n_total=160)
    B, steps, stride = 6, 44, 12
    torch.manual_seed(0)
    g = torch.Generator().manual_seed(123 + layers)
    lens0 = torch.randint(30, 70, (B,), generator=g).numpy().astype(np.int32)
    loop = DecodeLoop(cfg["h_q"], cfg["h_kv"], cfg["d"], cfg["b"], cfg["n_total"], cfg["N_max"], stride,
                      layers=layers, dtype=torch.bfloat16, window=cfg["w"], async_compress=async_compress,
                      decode_rho=decode_rho)
    loop.add_sequences(lens0)
    assert loop.use_rho == decode_rho
    # synthetic prefill: random rows in every block the sequences hold
    loop.K.copy_(zp_inputs.normal(tuple(loop.K.shape), 7, "bf16").cuda())
    loop.V.copy_(zp_inputs.normal(tuple(loop.V.shape), 8, "bf16").cuda())
    ora = OracleLoop(cfg, loop.K.float().cpu().numpy(), loop.V.float().cpu().numpy(), loop.table, loop.lens)
    total_swaps, compressions = 0, 0
    for step in range(steps):
        q = zp_inputs.normal((layers, B, cfg["h_q"], cfg["d"]), 1000 + step, "bf16")
        kn = zp_inputs.normal((layers, B, cfg["h_kv"], cfg["d"]), 2000 + step, "bf16")
        vn = zp_inputs.normal((layers, B, cfg["h_kv"], cfg["d"]), 3000 + step, "bf16")
        if async_compress:
            loop.drain()  # the oracle has no overlap: keep both sides in the same state
        trig = loop.step(q.cuda(), kn.cuda(), vn.cuda())
        torch.cuda.synchronize()
        out_ref, trig_ref = ora.step(q.float().numpy(), kn.float().numpy(), vn.float().numpy())
        assert sorted(int(x) for x in trig) == trig_ref
        got = loop.out.float().cpu().numpy()
        np.testing.assert_allclose(got, out_ref, **TOL_OUT["bf16"])
        if trig:
            seqs, keep = loop.last_keep
            keep = keep.cpu().numpy()
            for i, s in enumerate(seqs):
                total_swaps += ora.compress(int(s), keep[:, i])
                compressions += 1
            loop.drain()
            torch.cuda.synchronize()
            # state after compression: tables, lengths, caches of the compressed rows
            assert np.array_equal(loop.table, ora.table)
            assert np.array_equal(loop.lens, ora.lens)
            Kg = loop.K.float().cpu().numpy()
            Vg = loop.V.float().cpu().numpy()
            for s in seqs:
                for blk in ora.table[s, : cfg["N_max"] - 1]:
                    assert np.array_equal(Kg[:, blk], ora.K[:, blk])
                    assert np.array_equal(Vg[:, blk], ora.V[:, blk])
                    np.testing.assert_allclose(loop.F[:, blk].cpu().numpy(), ora.F[:, blk], rtol=1e-3, atol=1e-9)
        assert loop.pool.num_free == int((ora.ref == 0).sum())
    assert zp_device_clean()
    assert compressions >= B  # every sequence compressed at least once
    print("compressions", compressions, "reported tie swaps", total_swaps)


def zp_device_clean():
    import compressed_paged_kv_zp_gb300 as zp
    return zp.zp_device_status() == (0, 0)
