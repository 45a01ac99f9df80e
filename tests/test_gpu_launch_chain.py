"""Decode followed at once by the compression call on the same stream.

The decode kernel lets its dependents launch early, and the compression's two
kernels are launched as programmatic dependents: their CTAs may start while
the preceding kernel still runs, and they read what it writes (the score rows
of the window score, X and the row sums) only after waiting for it
(griddepcontrol.wait).  These tests check that the overlap changes nothing:
decode immediately followed by zp_compress_layers leaves bit for bit the
state of the same two calls with a device synchronisation between them, over
several repetitions; and the keep sets of sampled compressing sequences match
the oracle fed the decode's score rows.
"""
import pytest
import torch

import oracle
import zp_inputs
from oracle import pipeline
from tests.gpu_util import keep_sets_match

pytestmark = pytest.mark.gpu

B, H_Q, H_KV, D, BS, N_MAX, W = 64, 32, 8, 128, 16, 8, 16


def _setup():
    g = torch.Generator().manual_seed(4242)
    lens = (torch.randint(1024, 4097, (B,), generator=g) // BS * BS).tolist()
    c = zp_inputs.make_paged_case(4242, B, H_Q, H_KV, D, BS, lens=lens, dtype="bf16")
    zp_inputs.plant_duplicates(c, 4243)
    comp = list(range(0, B, 4))  # the compressing sequences (their score rows: their batch index)
    return c, comp


def _run(zp, c, comp, K0, V0, F0, chained, shared_ws=False):
    dev = torch.device("cuda")
    k = (N_MAX - 1) * BS
    desc = zp.cache_desc(H_Q, H_KV, D, BS, c.n_total, torch.bfloat16)
    K, V, F = K0.clone(), V0.clone(), F0.clone()
    q = c.q.to(dev)
    table = c.block_table.to(dev)
    lens = c.seq_lens.to(dev)
    out = torch.empty_like(q)
    S = torch.zeros(B, H_KV, table.shape[1] * BS, device=dev)
    idx = torch.tensor(comp, dtype=torch.long)
    c_table = c.block_table[idx].contiguous().to(dev)
    c_lens = c.seq_lens[idx].contiguous().to(dev)
    rows = idx.to(torch.int32).to(dev)
    first = torch.tensor([i % 2 for i in range(len(comp))], dtype=torch.uint8, device=dev)
    targets = c_table[:, : N_MAX - 1].contiguous()  # in place: the sequences' own blocks
    keep = torch.empty(len(comp), H_KV, k, dtype=torch.int32, device=dev)
    Lmax = int(c_lens.max())
    params = zp.score_params(window=W)
    ws_dec = ws_comp = None
    if shared_ws:
        # one scratch buffer for both calls, which stream order makes legal:
        # the compression may start while the decode drains and must not
        # store into it before the decode has completed
        n_ws = max(zp.zp_decode_workspace_size(desc, B, table.shape[1]),
                   zp.zp_compress_workspace_size(desc, len(comp), Lmax, 1))
        ws_dec = ws_comp = torch.zeros(n_ws, dtype=torch.uint8, device=dev)
    zp.zp_paged_decode_attn(desc, q, K, V, table, lens, out, score_accum=S, window=W, workspace=ws_dec)
    S_after_decode = None
    if not chained:
        torch.cuda.synchronize()
        S_after_decode = S.clone()
    zp.zp_compress_layers(desc, params, K, V, c_table, c_lens, first, S, F, targets, k, keep, Lmax, rows=rows,
                          workspace=ws_comp)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    return dict(out=out, S=S, K=K, V=V, F=F, keep=keep), S_after_decode, first


def test_decode_then_compression_without_sync_is_bit_exact():
    import compressed_paged_kv_zp_gb300 as zp
    c, comp = _setup()
    K0 = c.k_cache[0].contiguous().cuda()
    V0 = c.v_cache[0].contiguous().cuda()
    F0 = (torch.rand(c.n_total, BS, H_KV, generator=torch.Generator().manual_seed(7)) * 1e-3).cuda()
    ref, S_dec, first = _run(zp, c, comp, K0, V0, F0, chained=False)
    for _ in range(4):
        got, _, _ = _run(zp, c, comp, K0, V0, F0, chained=True)
        for name in ref:
            assert torch.equal(got[name], ref[name]), name
    # the keep sets of sampled compressing sequences against the oracle, fed the
    # score rows the decode left
    k = (N_MAX - 1) * BS
    prm = pipeline.ScoreParams(window=W)
    Kf = K0.float().cpu().numpy()
    swaps = 0
    for i in (0, len(comp) // 2, len(comp) - 1):
        s = comp[i]
        L = int(c.seq_lens[s])
        Fref = F0.double().cpu().numpy()
        sref = pipeline.final_scores(S_dec[s, :, :L].double().cpu().numpy(), Kf, Fref, c.block_table[s].numpy(),
                                     L, BS, bool(first[i]), prm)
        kp = ref["keep"][i].cpu().numpy()
        for h in range(H_KV):
            swaps += keep_sets_match(kp[h], oracle.topk_keep(sref[h], k)[0], sref[h], k, L)
    print("reported near-tie swaps:", swaps)


def test_compression_sharing_the_decode_scratch_is_bit_exact():
    """The compression handed the decode's own scratch buffer (reuse that stream
    order allows) and chained without a synchronisation leaves the state of the
    synchronised pair, bit for bit."""
    import compressed_paged_kv_zp_gb300 as zp
    c, comp = _setup()
    K0 = c.k_cache[0].contiguous().cuda()
    V0 = c.v_cache[0].contiguous().cuda()
    F0 = (torch.rand(c.n_total, BS, H_KV, generator=torch.Generator().manual_seed(8)) * 1e-3).cuda()
    ref, _, _ = _run(zp, c, comp, K0, V0, F0, chained=False)
    for _ in range(8):
        got, _, _ = _run(zp, c, comp, K0, V0, F0, chained=True, shared_ws=True)
        for name in ref:
            assert torch.equal(got[name], ref[name]), name
