"""GPU parity of the all-pairs ("flash") redundancy [Zipage App. C.5, Alg. 3]:
the row sums rho of the thresholded cosine matrix, read from the scoring
workspace after zp_score_tokens, against the oracle's rho of every (sequence,
kv head), or of sampled rows where the full matrix is too large for the
oracle.  Near-duplicate keys are planted inside blocks and far apart so that
the per-column zeroing acts within and across tiles and work items; cosines
of unrelated Gaussian keys stay far from the threshold, so every threshold
decision is unambiguous.

Layout relied on: the scoring workspace holds X [n][h_kv][Lmax] (fp32) and
then, 256-byte aligned, rho [n][h_kv][Lmax].
"""
import numpy as np
import pytest
import torch

import oracle
import zp_inputs
from oracle import pipeline
from tests.gpu_util import TOL_SCORE, DeviceCase

pytestmark = pytest.mark.gpu

RHO_TOL = dict(rtol=1e-4, atol=2e-3)  # fp32 row sums of up to 32k cosines


@pytest.fixture(scope="module")
def zp():
    import compressed_paged_kv_zp_gb300 as m
    return m


def _plant_far(keys_flat, phys, L, rng, count, lo, hi, noise=0.05):
    """Near-copies of earlier tokens lo..hi positions back, in place (numpy)."""
    h_kv, d = keys_flat.shape[1], keys_flat.shape[2]
    if L <= lo + 1:
        return
    dsts = rng.choice(np.arange(lo + 1, L), size=min(count, L - lo - 1), replace=False)
    for dst in dsts:
        src = dst - int(rng.integers(lo, min(hi, dst) + 1))
        keys_flat[phys[dst]] = keys_flat[phys[src]] + noise * rng.standard_normal((h_kv, d)).astype(np.float32)


def _case(seed, lens, h_kv, d, dtype, far=True, zero_key=None):
    B, b = len(lens), 16
    c = zp_inputs.make_paged_case(seed, B, 4 * h_kv, h_kv, d, b, lens=lens, dtype=dtype)
    zp_inputs.plant_duplicates(c, seed + 1)
    rng = np.random.default_rng(seed + 2)
    K = c.k_cache[0].float().numpy()
    flat = K.reshape(-1, h_kv, d)
    for s, L in enumerate(lens):
        t = np.arange(L)
        phys = c.block_table[s].numpy()[t // b] * b + t % b
        if far:
            _plant_far(flat, phys, L, rng, max(L // 25, 1), 40, 3000)
        if zero_key is not None and zero_key < L:
            flat[phys[zero_key]] = 0.0
    c.k_cache[0] = torch.from_numpy(K).to(c.k_cache.dtype)
    return c


def _run_rho(zp, c, p, lightning=False):
    """zp_score_tokens with the all-pairs redundancy; returns (rho, scores)."""
    dt = torch.bfloat16 if c.dtype == "bf16" else torch.float32
    desc = zp.cache_desc(c.h_q, c.h_kv, c.d, c.b, c.n_total, dt)
    dc = DeviceCase(c)
    n, h_kv = c.B, c.h_kv
    Lmax = int(c.seq_lens.max())
    S = torch.full((n, h_kv, Lmax), 0.01, device="cuda")
    F = torch.zeros(c.n_total, c.b, h_kv, device="cuda")
    first = torch.ones(n, dtype=torch.uint8, device="cuda")
    scores = torch.full((n, h_kv, Lmax), -3.0, device="cuda")
    ws = torch.empty(zp.zp_score_workspace_size(desc, n, Lmax), dtype=torch.uint8, device="cuda")
    params = zp.score_params(window=1, lightning=lightning, threshold=p)
    zp.zp_score_tokens(desc, params, dc.K[0], dc.table, dc.lens, first, S, F, scores, workspace=ws)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    off = (n * h_kv * Lmax * 4 + 255) // 256 * 256
    rho = ws[off:off + n * h_kv * Lmax * 4].view(torch.float32).view(n, h_kv, Lmax).cpu().numpy()
    return rho, scores.cpu().numpy()


@pytest.mark.parametrize("name,lens,h_kv,d,dtype,p", [
    ("qwen_d128", [304, 800, 1504], 8, 128, "bf16", 0.9),
    ("ragged_d64", [1, 17, 100, 777, 2000], 2, 64, "bf16", 0.9),
    ("every_pair_a_hit", [5, 130, 530], 2, 64, "bf16", -0.95),
    ("tiny_fp32", [80, 117, 150, 96], 2, 64, "f32", 0.9),
    ("fp32_d128_neg_p", [33, 200], 2, 128, "f32", -0.95),
])
def test_all_pairs_rho_matches_oracle(zp, name, lens, h_kv, d, dtype, p):
    """rho of every (sequence, kv head) against orc_redundancy_rho (fp64 over
    the explicit L x L matrix); with p = -0.95 every pair is above the
    threshold, so every column's newest row is zeroed (exact path everywhere);
    a zero-norm key is included."""
    c = _case(1100 + len(name), lens, h_kv, d, dtype, zero_key=3)
    rho, _ = _run_rho(zp, c, p)
    K0 = c.k_cache[0].float().numpy()
    for s, L in enumerate(lens):
        keys = pipeline.gather_rows(K0, c.block_table[s].numpy(), L, c.b)
        for h in range(h_kv):
            want = oracle.redundancy_rho(np.ascontiguousarray(keys[:, h]), c.b, p, 0)
            np.testing.assert_allclose(rho[s, h, :L], want, **RHO_TOL, err_msg="%s s=%d h=%d" % (name, s, h))


def test_all_pairs_final_scores_fp32(zp):
    """fp32 keys through the whole scoring call with the all-pairs redundancy
    (tiny workload, every flag of the redundancy path) at the fp32 score
    tolerance."""
    c = _case(1120, [80, 117, 150, 96], 2, 64, "f32")
    dc = DeviceCase(c)
    desc = zp.cache_desc(c.h_q, c.h_kv, c.d, c.b, c.n_total, torch.float32)
    lens = c.seq_lens.tolist()
    Lmax = max(lens)
    rng = np.random.default_rng(1121)
    S0 = (rng.random((c.B, c.h_kv, Lmax)) / 100).astype(np.float32)
    K0 = c.k_cache[0].float().numpy()
    for w, pool_policy, use_global in ((16, 1, True), (4, 2, False), (8, 0, True)):
        params = zp.score_params(window=w, lightning=False, pool_policy=pool_policy, use_global=use_global,
                                 tau=0.05)
        prm = pipeline.ScoreParams(window=w, lightning=False, pool_policy=pool_policy, use_global=use_global,
                                   tau=0.05)
        S = torch.from_numpy(S0.copy()).cuda()
        F = torch.zeros(c.n_total, c.b, c.h_kv, device="cuda")
        first = torch.ones(c.B, dtype=torch.uint8, device="cuda")
        scores = torch.full((c.B, c.h_kv, Lmax), -3.0, device="cuda")
        zp.zp_score_tokens(desc, params, dc.K[0], dc.table, dc.lens, first, S, F, scores)
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        got = scores.cpu().numpy()
        for s, L in enumerate(lens):
            Fref = np.zeros((c.n_total, c.b, c.h_kv))
            want = pipeline.final_scores(S0[s, :, :L].astype(np.float64), K0, Fref, c.block_table[s].numpy(), L,
                                         c.b, True, prm)
            fin = np.isfinite(want)
            assert np.array_equal(fin, np.isfinite(got[s, :, :L]))
            np.testing.assert_allclose(got[s, :, :L][fin], want[fin], **TOL_SCORE["f32"])


def test_all_pairs_rho_spanning_work_items(zp):
    """One 8800-token sequence (two column work items for the first row
    super-tiles), duplicates up to 8000 tokens apart; rho at sampled rows (the
    rows of planted pairs, the super-tile and item boundaries, random rows)
    against the row-wise oracle."""
    L, h_kv, d = 8800, 1, 64
    c = _case(1130, [L], h_kv, d, "bf16", far=False)
    rng = np.random.default_rng(1131)
    K = c.k_cache[0].float().numpy()
    flat = K.reshape(-1, h_kv, d)
    t = np.arange(L)
    phys = c.block_table[0].numpy()[t // c.b] * c.b + t % c.b
    pairs = []
    for _ in range(60):
        dst = int(rng.integers(8200, L))
        src = dst - int(rng.integers(500, 8100))
        flat[phys[dst]] = flat[phys[src]] + 0.05 * rng.standard_normal((h_kv, d)).astype(np.float32)
        pairs += [src, dst]
    c.k_cache[0] = torch.from_numpy(K).to(torch.bfloat16)
    rho, _ = _run_rho(zp, c, 0.9)
    keys = pipeline.gather_rows(c.k_cache[0].float().numpy(), c.block_table[0].numpy(), L, c.b)[:, 0]
    rows = sorted(set(pairs + [0, 511, 512, 1023, 8191, 8192, 8703, 8704, L - 1]
                      + rng.integers(0, L, 40).tolist()))
    want = oracle.redundancy_rho_rows(np.ascontiguousarray(keys), 0.9, np.array(rows, dtype=np.int32))
    np.testing.assert_allclose(rho[0, 0, rows], want, **RHO_TOL)
    assert np.abs(want).max() > 1.0


def test_all_pairs_rho_long_prefill_full_size(zp):
    """The long-prefill workload at full size: 16 sequences x 32768 tokens x 8
    kv heads, head_dim 128, bf16, keys drawn on the device, 200 near-copies per
    sequence planted up to 30000 tokens apart.  rho at sampled rows of four
    (sequence, kv head) pairs against the row-wise oracle (the full 32k x 32k
    matrix per head is out of the oracle's reach)."""
    B, h_kv, d, b, L = 16, 8, 128, 16, 32768
    c = zp_inputs.make_paged_case(1140, B, 32, h_kv, d, b, lens=[L] * B, dtype="bf16", device="cuda")
    K = c.k_cache[0]
    g = torch.Generator(device="cuda").manual_seed(1141)
    table = c.block_table.cuda().long()
    planted = {}
    rng = np.random.default_rng(1142)
    for s in range(B):
        dst = torch.from_numpy(rng.choice(np.arange(30000, L), 200, replace=False)).cuda()
        src = dst - torch.from_numpy(rng.integers(1000, 30000, 200)).cuda()
        kd = K[table[s, dst // b], dst % b]
        ks = K[table[s, src // b], src % b].float()
        K[table[s, dst // b], dst % b] = (ks + 0.05 * torch.randn(ks.shape, generator=g, device="cuda")).to(kd.dtype)
        planted[s] = (src.cpu().numpy(), dst.cpu().numpy())
    desc = zp.cache_desc(32, h_kv, d, b, c.n_total, torch.bfloat16)
    lens = c.seq_lens.cuda()
    tab = c.block_table.cuda()
    S = torch.full((B, h_kv, L), 0.01, device="cuda")
    F = torch.zeros(c.n_total, b, h_kv, device="cuda")
    first = torch.ones(B, dtype=torch.uint8, device="cuda")
    scores = torch.empty(B, h_kv, L, device="cuda")
    ws = torch.empty(zp.zp_score_workspace_size(desc, B, L), dtype=torch.uint8, device="cuda")
    zp.zp_score_tokens(desc, zp.score_params(window=16, lightning=False), K, tab, lens, first, S, F, scores,
                       workspace=ws)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    off = (B * h_kv * L * 4 + 255) // 256 * 256
    rho = ws[off:off + B * h_kv * L * 4].view(torch.float32).view(B, h_kv, L)
    for s, h in ((0, 0), (5, 3), (11, 7), (15, 1)):
        keys = K[table[s, torch.arange(L, device="cuda") // b], torch.arange(L, device="cuda") % b, h]
        keys = keys.float().cpu().numpy()
        src, dst = planted[s]
        rows = sorted(set(src[:6].tolist() + dst[:6].tolist() + [0, 511, 512, 8191, 8192, L - 1]))
        want = oracle.redundancy_rho_rows(np.ascontiguousarray(keys), 0.9, np.array(rows, dtype=np.int32))
        np.testing.assert_allclose(rho[s, h, rows].cpu().numpy(), want, **RHO_TOL, err_msg="s=%d h=%d" % (s, h))
