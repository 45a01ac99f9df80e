"""Compression at full workload sizes, through the C ABI in the order the
engine launches it: explicit window score -> final scores -> top-k ->
compaction.

* Long prefill: 16 sequences of 32768 tokens, 32q/8kv/128 bf16, b = 16,
  N_max = 128 (k = 2032), window of 16 queries, first compression (global
  score F <- S, pooling, lightning redundancy), Gaussian keys and the
  duplicate-planted variant (10% of tokens a near-copy of an earlier token of
  their block).
* Qwen3-8B layer batch: 64 sequences of 1024..4096 tokens rounded down to a
  whole block, N_max = 8 (k = 112); half of them at their first compression,
  the others at a later one with a random global score F.
Checked for every sequence: keep sets ascending, complete, inside [0, L), the
window kept; every moved K/V row bit-exact against the row its keep index
names, and F of the new slot equal to that token's global score; no device
error.  Against the oracle on sampled sequences
(all kv heads): final scores (1e-3 relative), keep sets (exact up to reported
near-ties).  Inputs are drawn on the device from seeded generators; the oracle
reads them back before any kernel runs.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import pipeline
from tests.gpu_util import TOL_SCORE, keep_sets_match

pytestmark = pytest.mark.gpu


def _dev_normal(shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(*shape, generator=g, device="cuda", dtype=torch.float32)


def _paged_case(seed, lens, h_kv, d, b, dup):
    """K, V [1][n_total][b][h_kv][d] bf16 with each sequence's blocks at a
    seeded permutation of the pool; table int32 [n][stride]."""
    g = torch.Generator().manual_seed(seed)
    nb = [(L + b - 1) // b for L in lens]
    n_total = sum(nb)
    stride = max(nb)
    perm = torch.randperm(n_total, generator=g).numpy().astype(np.int32)
    table = np.full((len(lens), stride), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(nb):
        table[s, :n] = perm[cur:cur + n]
        cur += n
    K = _dev_normal((1, n_total, b, h_kv, d), seed + 1)
    V = _dev_normal((1, n_total, b, h_kv, d), seed + 2).to(torch.bfloat16)
    if dup:
        # in the sequence's own order: 10% of tokens t become k_{t-delta} + 0.05 eps,
        # delta in [1, t mod b] so the original is in the same block
        Kf = K.view(n_total * b, h_kv, d)
        for s, L in enumerate(lens):
            t = np.arange(L)
            phys = table[s, t // b].astype(np.int64) * b + t % b
            pick = t[(t % b > 0) & (torch.rand(L, generator=g).numpy() < 0.1)]
            if not len(pick):
                continue
            delta = 1 + (torch.rand(len(pick), generator=g).numpy() * (pick % b)).astype(np.int64)
            src = torch.from_numpy(phys[pick - delta]).cuda()
            dst = torch.from_numpy(phys[pick]).cuda()
            eps = _dev_normal((len(pick), h_kv, d), seed + 3 + s)
            Kf[dst] = Kf[src] + 0.05 * eps
    return K.to(torch.bfloat16), V, table


def _seq_blocks(t, table_row, L, b):
    """float32 numpy copy of one sequence's blocks of a paged device tensor
    [n_total][b][...], and the renumbered table row."""
    nb = (L + b - 1) // b
    blk = torch.from_numpy(table_row[:nb].astype(np.int64)).to(t.device)
    return t.index_select(0, blk).float().cpu().numpy(), np.arange(nb, dtype=np.int32)


def _run(zp, lens, N_max, dup, first_mask, seed, n_sample):
    h_q, h_kv, d, b, w = 32, 8, 128, 16, 16
    n = len(lens)
    k = (N_max - 1) * b
    K, V, table = _paged_case(seed, lens, h_kv, d, b, dup)
    n_total = K.shape[1]
    desc = zp.cache_desc(h_q, h_kv, d, b, n_total, torch.bfloat16)
    qw = _dev_normal((n, w, h_q, d), seed + 7).to(torch.bfloat16)
    F = torch.rand(n_total, b, h_kv, generator=torch.Generator(device="cuda").manual_seed(seed + 8),
                   device="cuda") * 1e-3
    first = torch.from_numpy(first_mask.astype(np.uint8)).cuda()
    table_d = torch.from_numpy(table).cuda()
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    Lmax = max(lens)
    sample = list(np.linspace(0, n - 1, n_sample).astype(int))
    # the oracle's copies of the sampled sequences' inputs, before any kernel runs
    ins = {}
    for s in sample:
        Ks, tab = _seq_blocks(K[0], table[s], lens[s], b)
        Fs, _ = _seq_blocks(F, table[s], lens[s], b)
        ins[s] = (qw[s].float().cpu().numpy(), Ks, Fs.astype(np.float64), tab)
    S = torch.empty(n, h_kv, Lmax, device="cuda")
    zp.zp_window_score(desc, qw, K[0], table_d, lens_d, S)
    scores = torch.empty(n, h_kv, Lmax, device="cuda")
    prm = zp.score_params(window=w)
    zp.zp_score_tokens(desc, prm, K[0], table_d, lens_d, first, S, F, scores)
    keep = torch.empty(n, h_kv, k, dtype=torch.int32, device="cuda")
    ties = torch.zeros(n, h_kv, dtype=torch.int32, device="cuda")
    zp.zp_select_topk(scores, lens_d, k, keep, ties)
    K0, V0 = K.clone(), V.clone()
    targets = torch.from_numpy(np.ascontiguousarray(table[:, : N_max - 1])).cuda()
    zp.zp_compact_pages(desc, K, V, 0, 1, F, 0, table_d, targets, lens_d, keep, k, scores=S)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)

    # every sequence: keep sets and moved rows
    kp = keep.long()
    assert torch.all(kp[..., 1:] > kp[..., :-1])
    assert torch.all(kp[..., 0] >= 0)
    assert torch.all(kp[..., -1] < lens_d.long()[:, None])
    for s, L in enumerate(lens):
        win = torch.arange(L - w, L, device="cuda")
        assert torch.equal(kp[s, :, k - w:], win.expand(h_kv, w))  # the window survives in every head
        tb = torch.from_numpy(table[s].astype(np.int64)).cuda()
        src = tb[kp[s] // b] * b + kp[s] % b                  # [h_kv][k] source slots
        r = torch.arange(k, device="cuda")
        dst = (tb[r // b] * b + r % b)[None, :].expand(h_kv, k)  # rank r -> slot r of target r/b
        hh = torch.arange(h_kv, device="cuda")[:, None].expand(h_kv, k)
        Kv0, Kv = K0[0].view(-1, h_kv, d), K[0].view(-1, h_kv, d)
        Vv0, Vv = V0[0].view(-1, h_kv, d), V[0].view(-1, h_kv, d)
        assert torch.equal(Kv[dst, hh], Kv0[src, hh])
        assert torch.equal(Vv[dst, hh], Vv0[src, hh])
        # F of the new slot: the kept token's global score, left in the score row
        assert torch.equal(F.view(-1, h_kv)[dst, hh], S[s][hh, kp[s]])

    # sampled sequences against the oracle
    got_scores = scores.cpu().numpy()
    got_keep = keep.cpu().numpy()
    oprm = pipeline.ScoreParams(window=w)
    swaps = 0
    for s in sample:
        q_s, K_s, F_s, tab = ins[s]
        L = lens[s]
        Sref = oracle.window_score(q_s, K_s, tab, L, w)
        sref = pipeline.final_scores(Sref, K_s, F_s, tab, L, b, bool(first_mask[s]), oprm)
        np.testing.assert_allclose(got_scores[s, :, :L], sref, **TOL_SCORE["bf16"])
        for h in range(h_kv):
            kref = oracle.topk_keep(sref[h], k)[0]
            swaps += keep_sets_match(got_keep[s, h], kref, sref[h], k, L)
    return swaps, int(ties.sum())


@pytest.mark.parametrize("dup", [False, True])
def test_long_prefill_first_compression_16x32k(dup):
    import compressed_paged_kv_zp_gb300 as zp
    lens = [32768] * 16
    swaps, ties = _run(zp, lens, 128, dup, np.ones(16, dtype=bool), 1004 + 10 * dup, n_sample=2)
    print("reported near-tie swaps:", swaps, "device tie count:", ties)


def test_qwen_layer_batch_64_sequences():
    import compressed_paged_kv_zp_gb300 as zp
    g = torch.Generator().manual_seed(1002)
    lens = [int(x) // 16 * 16 for x in torch.randint(1024, 4097, (64,), generator=g)]
    first = np.arange(64) % 2 == 0
    swaps, ties = _run(zp, lens, 8, True, first, 1102, n_sample=4)
    print("reported near-tie swaps:", swaps, "device tie count:", ties)
