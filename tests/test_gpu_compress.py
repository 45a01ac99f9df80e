"""GPU parity of the compression step: scores, top-k keep sets, compaction.

* zp_score_tokens vs the oracle pipeline (gather + Alg. 2 + pooling +
  lightning redundancy + eq. 4 + window), first and later compressions,
  duplicate-planted keys so the similarity threshold fires;
* zp_select_topk vs the oracle on identical float scores: bit-exact, ties
  (pooling plateaus) included, L <= k and L = k + 1;
* zp_compact_pages vs Alg. 4 of the oracle: bit-exact bytes, in place and
  into fresh target blocks, several layers, F moved with the rows;
* end to end on the tiny and Qwen-shaped workloads: keep sets equal except for
  reported swaps among near-tied scores; retained count == (N_max - 1) * b.
"""
import numpy as np
import pytest
import torch

import oracle
import zp_inputs
from oracle import pipeline
from tests.gpu_util import TOL_SCORE, DeviceCase, gather_slots, keep_sets_match

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zp():
    import compressed_paged_kv_zp_gb300 as m
    return m


def _desc(zp, c):
    return zp.cache_desc(c.h_q, c.h_kv, c.d, c.b, c.n_total,
                         torch.bfloat16 if c.dtype == "bf16" else torch.float32)


def _block_aligned_case(seed, B, h_q, h_kv, d, b, lo, hi, dtype, dup=False, spare=0):
    g = torch.Generator().manual_seed(seed)
    lens = (torch.randint(lo, hi + 1, (B,), generator=g) // b * b).clamp(min=b).tolist()
    c = zp_inputs.make_paged_case(seed, B, h_q, h_kv, d, b, lens=lens, dtype=dtype, spare_blocks=spare)
    if dup:
        zp_inputs.plant_duplicates(c, seed + 1)
    return c


SCORE_CASES = [
    # name, B, h_q, h_kv, d, b, lo, hi, dtype, dup, first, prm
    ("tiny_first", 4, 8, 2, 64, 16, 80, 150, "f32", False, True, {}),
    ("tiny_dup_later", 4, 8, 2, 64, 16, 80, 150, "f32", True, False, {}),
    ("tiny_nosim_everypool", 3, 8, 2, 64, 16, 60, 100, "f32", False, False,
     dict(use_similarity=False, pool_policy=2)),
    ("tiny_noglobal", 3, 8, 2, 64, 16, 60, 100, "f32", True, True, dict(use_global=False, pool_kernel=3)),
    ("qwen_dup_first", 6, 32, 8, 128, 16, 200, 900, "bf16", True, True, {}),
    ("qwen_later_w8", 5, 32, 8, 128, 16, 200, 600, "bf16", True, False, dict(window=8)),
]


@pytest.mark.parametrize("name,B,h_q,h_kv,d,b,lo,hi,dtype,dup,first,prm", SCORE_CASES)
def test_score_tokens_matches_oracle(zp, name, B, h_q, h_kv, d, b, lo, hi, dtype, dup, first, prm):
    seed = 300 + [x[0] for x in SCORE_CASES].index(name)
    c = _block_aligned_case(seed, B, h_q, h_kv, d, b, lo, hi, dtype, dup)
    dc = DeviceCase(c)
    P = pipeline.ScoreParams(**prm)
    params = zp.score_params(window=P.window, use_global=P.use_global, alpha=P.alpha,
                             pool_kernel=P.pool_kernel, pool_policy=P.pool_policy,
                             use_similarity=P.use_similarity, lightning=P.lightning, threshold=P.p,
                             lam=P.lam, tau=P.tau)
    rng = np.random.default_rng(seed)
    # attention-score rows in a larger table, reached through a row map
    Lrow = int(c.seq_lens.max()) + 3
    S0 = (rng.random((B + 2, h_kv, Lrow)) / 50).astype(np.float32)
    rows = np.array([(B + 1 - s) for s in range(B)], dtype=np.int32)
    S = torch.from_numpy(S0).cuda()
    F0 = (rng.random((c.n_total, b, h_kv)) / 40).astype(np.float32)
    F = torch.from_numpy(F0).cuda()
    Lmax = int(c.seq_lens.max()) + 5
    out = torch.full((B, h_kv, Lmax), -7.0, device="cuda")
    first_t = torch.full((B,), 1 if first else 0, dtype=torch.uint8, device="cuda")
    zp.zp_score_tokens(_desc(zp, c), params, dc.K[0], dc.table, dc.lens, first_t, S, F, out,
                       rows=torch.from_numpy(rows).cuda())
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    got = out.cpu().numpy()
    S_after = S.cpu().numpy().astype(np.float64)
    F_ref = F0.astype(np.float64)
    K = dc.np_k()
    for s in range(B):
        L = int(c.seq_lens[s])
        S_seq = S0[rows[s], :, :L].astype(np.float64)
        ref = pipeline.final_scores(S_seq, K, F_ref, c.block_table[s].numpy(), L, b, first, P)
        fin = np.isfinite(ref)
        assert np.array_equal(np.isinf(got[s, :, :L]), ~fin)
        np.testing.assert_allclose(got[s, :, :L][fin], ref[fin], **TOL_SCORE["f32"])
        assert np.all(got[s, :, L:] == -7.0)  # untouched beyond L
        # the row now holds the global score (what F of the kept tokens receives)
        want = gather_slots(F_ref, c.block_table[s].numpy(), L, b) if P.use_global else S_seq
        np.testing.assert_allclose(S_after[rows[s], :, :L], want, rtol=1e-6, atol=0)
        assert np.array_equal(S_after[rows[s], :, L:], S0[rows[s], :, L:])
    assert np.array_equal(S_after[0], S0[0])  # a row no sequence maps to
    assert np.array_equal(F.cpu().numpy(), F0)  # F is only read


TOPK_CASES = [(L, k) for L in (1, 47, 48, 49, 160, 1000, 4099) for k in (48, 112)] + [(32768, 2032)]


@pytest.mark.parametrize("L,k", TOPK_CASES)
def test_topk_bit_exact(zp, L, k):
    rng = np.random.default_rng(L * 7 + k)
    n, h_kv = 3, 2
    Lmax = L + 3
    sc = rng.random((n, h_kv, Lmax)).astype(np.float32)
    sc[0, 0, : L // 2] = 0.25  # a plateau (ties) crossing the threshold
    sc[1, 1] = np.round(sc[1, 1] * 8) / 8  # few distinct values
    sc[2, 0, L - 16:L] = np.inf  # window
    sc[2, 1, :L] = -sc[2, 1, :L]  # negative scores
    lens = np.array([L, max(L - 1, 1), L], dtype=np.int32)
    keep = torch.full((n, h_kv, k), -9, dtype=torch.int32, device="cuda")
    ties = torch.full((n, h_kv), -1, dtype=torch.int32, device="cuda")
    zp.zp_select_topk(torch.from_numpy(sc).cuda(), torch.from_numpy(lens).cuda(), k, keep, ties)
    torch.cuda.synchronize()
    got = keep.cpu().numpy()
    for s in range(n):
        for h in range(h_kv):
            ref, _, cnt = oracle.topk_keep(sc[s, h, : lens[s]].astype(np.float64), k)
            assert np.array_equal(got[s, h], ref), (s, h)
            assert cnt == min(k, lens[s])
    t = ties.cpu().numpy()
    if lens[1] > k:
        assert t[1, 1] > 1  # the quantised row has a split tie at the threshold
    if lens[1] <= k:
        assert t[1, 1] == 0


def _compaction_setup(zp, seed, layers, fresh_targets):
    b, h_kv, d, h_q = 16, 8, 128, 32
    N_max = 4
    k = (N_max - 1) * b
    lens = [4 * b, 7 * b, 5 * b]
    c = zp_inputs.make_paged_case(seed, 3, h_q, h_kv, d, b, lens=lens, dtype="bf16", layers=layers,
                                  spare_blocks=16)
    dc = DeviceCase(c)
    rng = np.random.default_rng(seed)
    keep = np.full((layers, 3, h_kv, k), -1, dtype=np.int32)
    for l in range(layers):
        for s, L in enumerate(lens):
            for h in range(h_kv):
                keep[l, s, h] = np.sort(rng.choice(L, k, replace=False))
    free = c.free_blocks.numpy()
    if fresh_targets:
        tgt = free[: 3 * (N_max - 1)].reshape(3, N_max - 1)
    else:
        tgt = c.block_table.numpy()[:, : N_max - 1].copy()
    F = torch.from_numpy(rng.random((layers, c.n_total, b, h_kv)).astype(np.float32)).cuda()
    # the global scores zp_score_tokens leaves in the score rows
    S = torch.from_numpy(rng.random((layers, 3, h_kv, 8 * b + 5)).astype(np.float32)).cuda()
    return c, dc, keep, tgt, F, S, k


@pytest.mark.parametrize("layers,fresh", [(1, False), (3, False), (2, True)])
def test_compaction_bit_exact_vs_alg4(zp, layers, fresh):
    c, dc, keep, tgt, F, S, k = _compaction_setup(zp, 500 + layers, layers, fresh)
    Kraw = dc.K.view(torch.int16).cpu().numpy().copy()
    Vraw = dc.V.view(torch.int16).cpu().numpy().copy()
    F0 = F.cpu().numpy().copy()
    Srows = S.cpu().numpy()
    desc = _desc(zp, c)
    layer_stride = c.n_total * c.b * c.h_kv * c.d
    zp.zp_compact_pages(desc, dc.K, dc.V, layer_stride, layers, F, c.n_total * c.b * c.h_kv,
                        dc.table, torch.from_numpy(tgt).cuda(), dc.lens, torch.from_numpy(keep).cuda(), k,
                        scores=S)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    row = c.d * 2
    # Alg. 4 with F holding each sequence's global score at its own slots;
    # the library writes F only in the target slots, the rest stays as it was
    Fsrc = F0.copy()
    for s, L in enumerate(c.seq_lens.tolist()):
        t = np.arange(L)
        for l in range(layers):
            Fsrc[l, c.block_table[s].numpy()[t // c.b], t % c.b] = Srows[l, s, :, :L].T
    Fmoved = Fsrc.copy()
    for s, L in enumerate(c.seq_lens.tolist()):
        N = (L + c.b - 1) // c.b
        pipeline.compact_sequence([Kraw, Vraw, Fmoved], [row, row, 4], c.b, c.h_kv,
                                  c.block_table[s].numpy(), N, tgt[s], keep[:, s], L)
    Fwant = F0.copy()
    r = np.arange(k)
    for s in range(3):
        Fwant[:, tgt[s][r // c.b], r % c.b] = Fmoved[:, tgt[s][r // c.b], r % c.b]
    assert np.array_equal(dc.K.view(torch.int16).cpu().numpy(), Kraw)
    assert np.array_equal(dc.V.view(torch.int16).cpu().numpy(), Vraw)
    assert np.array_equal(F.cpu().numpy(), Fwant)


@pytest.mark.parametrize("shape", ["tiny", "qwen"])
def test_end_to_end_compression(zp, shape):
    """decode window -> scores -> top-k -> plan -> compaction, against the oracle."""
    if shape == "tiny":
        B, h_q, h_kv, d, b, N_max, dtype, lo, hi = 4, 8, 2, 64, 16, 4, "f32", 80, 150
    else:
        B, h_q, h_kv, d, b, N_max, dtype, lo, hi = 8, 32, 8, 128, 16, 8, "bf16", 200, 700
    w = 16
    c = _block_aligned_case(900 + len(shape), B, h_q, h_kv, d, b, lo, hi, dtype, dup=True, spare=B * N_max)
    dc = DeviceCase(c)
    desc = _desc(zp, c)
    S = torch.zeros(B, h_kv, c.block_table.shape[1] * b, device="cuda")
    # the last w steps of each sequence, queries from the seeded generator
    final = c.seq_lens.tolist()
    qw = zp_inputs.normal((B, w, h_q, d), 901, dtype)
    for u in range(w):
        lens_d = torch.tensor([L - w + u + 1 for L in final], dtype=torch.int32, device="cuda")
        q = qw[:, u].contiguous().cuda()
        zp.zp_paged_decode_attn(desc, q, dc.K[0], dc.V[0], dc.table, lens_d, torch.empty_like(q),
                                score_accum=S, window=w)
    F = torch.zeros(c.n_total, b, h_kv, device="cuda")
    Lmax = max(final)
    scores = torch.empty(B, h_kv, Lmax, device="cuda")
    first = torch.ones(B, dtype=torch.uint8, device="cuda")
    params = zp.score_params(window=w)
    zp.zp_score_tokens(desc, params, dc.K[0], dc.table, dc.lens, first, S, F, scores)
    k = (N_max - 1) * b
    keep = torch.empty(B, h_kv, k, dtype=torch.int32, device="cuda")
    zp.zp_select_topk(scores, dc.lens, k, keep)
    # host planner (no sharing): targets are the first N_max-1 blocks
    pool = zp.Pool(c.n_total)
    pool.alloc(c.n_total)  # everything in use; release what the table does not hold
    held = set(int(x) for x in c.block_table.flatten().tolist() if x >= 0)
    pool.release([i for i in range(c.n_total) if i not in held])
    tg = np.zeros((B, N_max - 1), dtype=np.int32)
    new_tables = []
    for s in range(B):
        N = final[s] // b
        plan = pool.plan_compaction(c.block_table[s, :N].tolist(), N_max)
        tg[s] = plan["targets"]
        new_tables.append(plan["new_table"])
        pool.release(plan["dropped"])
    zp.zp_compact_pages(desc, dc.K, dc.V, 0, 1, F, 0, dc.table, torch.from_numpy(tg).cuda(), dc.lens,
                        keep, k, scores=S)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    # ---- oracle, same steps
    K0 = c.k_cache[0].float().numpy()
    V0 = c.v_cache[0].float().numpy()
    P = pipeline.ScoreParams(window=w)
    swaps = 0
    Kg = dc.K[0].float().cpu().numpy()
    Vg = dc.V[0].float().cpu().numpy()
    kept_all = keep.cpu().numpy()
    for s in range(B):
        L = final[s]
        Sref = oracle.window_score(qw[s].float().numpy(), K0, c.block_table[s].numpy(), L, w)
        Fref = np.zeros((c.n_total, b, h_kv))
        sref = pipeline.final_scores(Sref, K0, Fref, c.block_table[s].numpy(), L, b, True, P)
        Fg = F.cpu().numpy()
        for h in range(h_kv):
            kref = oracle.topk_keep(sref[h], k)[0]
            swaps += keep_sets_match(kept_all[s, h], kref, sref[h], k, L)
            # retained rows: GPU-moved rows equal the source rows of the GPU keep set
            assert (kept_all[s, h] >= 0).sum() == k
            assert set(range(L - w, L)) <= set(kept_all[s, h].tolist())  # window kept
            src = kept_all[s, h]
            for r in range(0, k, 7):
                pos = src[r]
                sb, ss = c.block_table[s, pos // b], pos % b
                db, ds = tg[s, r // b], r % b
                assert np.array_equal(Kg[db, ds, h], K0[sb, ss, h])
                assert np.array_equal(Vg[db, ds, h], V0[sb, ss, h])
                # F of the new slot: the global score (first compression: S) of the kept token
                np.testing.assert_allclose(Fg[db, ds, h], Fref[sb, ss, h], **TOL_SCORE[dtype])
        assert len(new_tables[s]) == N_max
    print("reported tie swaps:", swaps)
    assert pool.num_free == c.n_total - B * N_max


@pytest.mark.parametrize("shape", ["tiny", "qwen", "long_rows"])
def test_compress_layer_matches_three_steps(zp, shape):
    """zp_compress_layers (scores, selection and move fused per (sequence, kv
    head), or the three steps for rows too long for shared memory) against the
    three separate calls on copies of the same state: scores within 1e-6
    relative, keep sets equal up to near-ties, every moved row bit-exact for
    the keep set each path chose; and its keep sets against the oracle."""
    if shape == "tiny":
        B, h_q, h_kv, d, N_max, dtype, lo, hi = 4, 8, 2, 64, 4, "f32", 80, 150
    elif shape == "qwen":
        B, h_q, h_kv, d, N_max, dtype, lo, hi = 8, 32, 8, 128, 8, "bf16", 200, 900
    else:
        B, h_q, h_kv, d, N_max, dtype, lo, hi = 2, 32, 8, 128, 128, "bf16", 29000, 30000
    b, w = 16, 16
    c = _block_aligned_case(950 + len(shape), B, h_q, h_kv, d, b, lo, hi, dtype, dup=True, spare=B * N_max)
    desc = _desc(zp, c)
    lens = c.seq_lens.tolist()
    Lmax = max(lens)
    k = (N_max - 1) * b
    rng = np.random.default_rng(951)
    S0 = (rng.random((B, h_kv, Lmax + 16)) / 100).astype(np.float32)
    F0 = (rng.random((c.n_total, b, h_kv)) / 80).astype(np.float32)
    first = torch.tensor([1, 0] * (B // 2), dtype=torch.uint8, device="cuda")
    free = c.free_blocks.numpy()
    tg = np.stack([free[i * (N_max - 1):(i + 1) * (N_max - 1)] if i % 2 else c.block_table[i, : N_max - 1].numpy()
                   for i in range(B)]).astype(np.int32)  # fresh targets for odd sequences, in place for even
    targets = torch.from_numpy(tg).cuda()
    params = zp.score_params(window=w)
    out = {}
    for path in ("three", "fused"):
        dc = DeviceCase(c)
        S = torch.from_numpy(S0.copy()).cuda()
        F = torch.from_numpy(F0.copy()).cuda()
        scores = torch.full((B, h_kv, Lmax), -5.0, device="cuda")
        keep = torch.empty(B, h_kv, k, dtype=torch.int32, device="cuda")
        if path == "three":
            zp.zp_score_tokens(desc, params, dc.K[0], dc.table, dc.lens, first, S, F, scores)
            zp.zp_select_topk(scores, dc.lens, k, keep)
            zp.zp_compact_pages(desc, dc.K, dc.V, 0, 1, F, 0, dc.table, targets, dc.lens, keep, k, scores=S)
        else:
            zp.zp_compress_layers(desc, params, dc.K[0], dc.V[0], dc.table, dc.lens, first, S, F, targets, k, keep,
                                 Lmax, scores_out=scores)
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        out[path] = (scores.cpu().numpy(), keep.cpu().numpy(), dc.K[0].float().cpu().numpy(),
                     dc.V[0].float().cpu().numpy(), F.cpu().numpy())
    s3, k3, K3, V3, F3 = out["three"]
    sf, kf, Kf, Vf, Ff = out["fused"]
    fin = np.isfinite(s3)
    assert np.array_equal(fin, np.isfinite(sf))
    np.testing.assert_allclose(sf[fin], s3[fin], rtol=1e-6, atol=1e-9)  # reduction order differs
    K0 = c.k_cache[0].float().numpy()
    V0 = c.v_cache[0].float().numpy()
    swaps = 0
    prm = pipeline.ScoreParams(window=w)
    for s in range(B):
        L = lens[s]
        for h in range(h_kv):
            swaps += keep_sets_match(kf[s, h], k3[s, h], s3[s, h], k, L)
            kept = kf[s, h]
            for r in range(0, min(k, L), 3):  # moved rows of the fused path
                pos = kept[r]
                sb, ss = c.block_table[s, pos // b], pos % b
                db, ds = tg[s, r // b], r % b
                assert np.array_equal(Kf[db, ds, h], K0[sb, ss, h])
                assert np.array_equal(Vf[db, ds, h], V0[sb, ss, h])
        if shape != "long_rows" or s == 0:  # the oracle, sampled for the long rows
            Fref = F0.astype(np.float64).copy()
            sref = pipeline.final_scores(S0[s, :, :L].astype(np.float64), K0, Fref, c.block_table[s].numpy(), L, b,
                                         bool(first[s]), prm)
            np.testing.assert_allclose(sf[s, :, :L][np.isfinite(sref)], sref[np.isfinite(sref)],
                                       **TOL_SCORE[dtype])
            for h in range(h_kv):
                swaps += keep_sets_match(kf[s, h], oracle.topk_keep(sref[h], k)[0], sref[h], k, L)
    print("reported near-tie swaps:", swaps)


@pytest.mark.parametrize("shape", ["qwen", "long_rows"])
def test_per_request_budgets(zp, shape):
    """Per-request budgets k_i = (N_i - 1) b given as a k_seq array, through
    zp_compress_layers and through zp_select_topk + zp_compact_pages: each
    keep row holds k_i positions then -1 up to the row stride k = max k_i;
    the keep sets equal the oracle's top-k_i up to reported near-ties; both
    paths agree; moved rows are bit-exact; no block outside the targets is
    written (the short budgets' unused target slots stay -1)."""
    b, w = 16, 16
    if shape == "qwen":
        B, h_q, h_kv, d, lo, hi = 6, 32, 8, 128, 200, 900
        N_i = np.array([2, 8, 5, 3, 8, 6], np.int32)
    else:  # rows too long for the fused kernel's shared memory: the three-step fallback
        B, h_q, h_kv, d, lo, hi = 2, 32, 8, 128, 29000, 30000
        N_i = np.array([128, 37], np.int32)
    N_max = int(N_i.max())
    c = _block_aligned_case(980 + len(shape), B, h_q, h_kv, d, b, lo, hi, "bf16", dup=True, spare=B * N_max)
    desc = _desc(zp, c)
    lens = c.seq_lens.tolist()
    Lmax = max(lens)
    k = (N_max - 1) * b
    k_i = (N_i - 1) * b
    rng = np.random.default_rng(981)
    S0 = (rng.random((B, h_kv, Lmax + 16)) / 100).astype(np.float32)
    F0 = (rng.random((c.n_total, b, h_kv)) / 80).astype(np.float32)
    first = torch.tensor([1, 0] * (B // 2), dtype=torch.uint8, device="cuda")
    free = c.free_blocks.numpy()
    tg = np.full((B, N_max - 1), -1, np.int32)
    for i in range(B):
        m = int(N_i[i]) - 1
        tg[i, :m] = free[i * (N_max - 1): i * (N_max - 1) + m] if i % 2 else c.block_table[i, :m].numpy()
    targets = torch.from_numpy(tg).cuda()
    k_seq = torch.from_numpy(k_i).cuda()
    params = zp.score_params(window=w)
    out = {}
    for path in ("three", "fused"):
        dc = DeviceCase(c)
        S = torch.from_numpy(S0.copy()).cuda()
        F = torch.from_numpy(F0.copy()).cuda()
        scores = torch.full((B, h_kv, Lmax), -5.0, device="cuda")
        keep = torch.full((B, h_kv, k), -7, dtype=torch.int32, device="cuda")
        if path == "three":
            zp.zp_score_tokens(desc, params, dc.K[0], dc.table, dc.lens, first, S, F, scores)
            zp.zp_select_topk(scores, dc.lens, k, keep, k_seq=k_seq)
            zp.zp_compact_pages(desc, dc.K, dc.V, 0, 1, F, 0, dc.table, targets, dc.lens, keep, k, scores=S,
                                k_seq=k_seq)
        else:
            zp.zp_compress_layers(desc, params, dc.K[0], dc.V[0], dc.table, dc.lens, first, S, F, targets, k, keep,
                                  Lmax, scores_out=scores, k_seq=k_seq)
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        out[path] = (scores.cpu().numpy(), keep.cpu().numpy(), dc.K[0].float().cpu().numpy(),
                     dc.V[0].float().cpu().numpy())
    s3, k3, K3, V3 = out["three"]
    sf, kf, Kf, Vf = out["fused"]
    K0 = c.k_cache[0].float().numpy()
    V0 = c.v_cache[0].float().numpy()
    written = set(tg[tg >= 0].tolist())
    untouched = np.array([x for x in range(c.n_total) if x not in written])
    prm = pipeline.ScoreParams(window=w)
    swaps = 0
    for s in range(B):
        L, ki = lens[s], int(k_i[s])
        for kp in (k3, kf):
            assert (kp[s, :, ki:] == -1).all()
            assert (kp[s, :, :min(ki, L)] >= 0).all()
        for h in range(h_kv):
            swaps += keep_sets_match(kf[s, h], k3[s, h], s3[s, h], ki, L)
            for Kx, Vx, kp in ((Kf, Vf, kf), (K3, V3, k3)):
                for r in range(0, min(ki, L), 5):
                    pos = kp[s, h, r]
                    sb, ss = c.block_table[s, pos // b], pos % b
                    db, ds = tg[s, r // b], r % b
                    assert np.array_equal(Kx[db, ds, h], K0[sb, ss, h])
                    assert np.array_equal(Vx[db, ds, h], V0[sb, ss, h])
        if shape != "long_rows" or s == 1:  # the oracle, sampled for the long rows
            Fref = F0.astype(np.float64).copy()
            sref = pipeline.final_scores(S0[s, :, :L].astype(np.float64), K0, Fref, c.block_table[s].numpy(), L, b,
                                         bool(first[s]), prm)
            for h in range(h_kv):
                swaps += keep_sets_match(kf[s, h], oracle.topk_keep(sref[h], ki)[0], sref[h], ki, L)
    for Kx, Vx in ((Kf, Vf), (K3, V3)):
        assert np.array_equal(Kx[untouched], K0[untouched])
        assert np.array_equal(Vx[untouched], V0[untouched])
    print("reported near-tie swaps:", swaps)


def test_compress_layers_several_layers_in_one_call(zp):
    """Three layers in one zp_compress_layers call (one launch per kernel,
    App. C.1) equal three single-layer calls: scores, keep sets, K, V and F
    bit-exact (the same arithmetic per layer)."""
    B, h_q, h_kv, d, b, N_max, layers = 5, 32, 8, 128, 16, 8, 3
    g = torch.Generator().manual_seed(960)
    lens = (torch.randint(200, 900, (B,), generator=g) // b * b).tolist()
    c = zp_inputs.make_paged_case(960, B, h_q, h_kv, d, b, lens=lens, dtype="bf16", layers=layers,
                                  spare_blocks=B * N_max)
    zp_inputs.plant_duplicates(c, 961)
    desc = _desc(zp, c)
    Lmax, k = max(lens), (N_max - 1) * b
    rng = np.random.default_rng(962)
    S0 = (rng.random((layers, B, h_kv, Lmax + 8)) / 100).astype(np.float32)
    F0 = (rng.random((layers, c.n_total, b, h_kv)) / 80).astype(np.float32)
    first = torch.tensor([0, 1, 0, 1, 0], dtype=torch.uint8, device="cuda")
    targets = c.block_table[:, : N_max - 1].contiguous().cuda()
    params = zp.score_params(window=16)
    res = {}
    for mode in ("one_call", "per_layer"):
        dc = DeviceCase(c)
        S = torch.from_numpy(S0.copy()).cuda()
        F = torch.from_numpy(F0.copy()).cuda()
        keep = torch.empty(layers, B, h_kv, k, dtype=torch.int32, device="cuda")
        scores = torch.full((layers, B, h_kv, Lmax), -5.0, device="cuda")
        if mode == "one_call":
            zp.zp_compress_layers(desc, params, dc.K, dc.V, dc.table, dc.lens, first, S, F, targets, k, keep, Lmax,
                                  scores_out=scores)
        else:
            for l in range(layers):
                zp.zp_compress_layers(desc, params, dc.K[l], dc.V[l], dc.table, dc.lens, first, S[l], F[l],
                                      targets, k, keep[l], Lmax, scores_out=scores[l])
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        res[mode] = [t.cpu() for t in (scores, keep, dc.K, dc.V, F, S)]
    for x, y in zip(res["one_call"], res["per_layer"]):
        assert torch.equal(x, y)


def test_all_pairs_redundancy_matches_oracle(zp):
    """The all-pairs ('flash') redundancy score [App. C.5, Alg. 3] on bf16 keys
    against the oracle's definition over the full L x L cosine matrix, with
    near-duplicates planted inside blocks and hundreds of tokens apart (so the
    per-column zeroing acts across tiles), through zp_score_tokens and through
    zp_compress_layers (keep sets and moved rows)."""
    B, h_q, h_kv, d, b, N_max = 3, 32, 8, 128, 16, 8
    lens = [304, 800, 1504]
    c = zp_inputs.make_paged_case(970, B, h_q, h_kv, d, b, lens=lens, dtype="bf16", spare_blocks=B * N_max)
    zp_inputs.plant_duplicates(c, 971)
    rng = np.random.default_rng(972)
    Kc = c.k_cache[0].float().numpy()
    for s, L in enumerate(lens):  # far-apart near-copies, in the sequence's own order
        t = np.arange(L)
        phys = c.block_table[s].numpy()[t // b] * b + t % b
        flat = Kc.reshape(-1, h_kv, d)
        pool = np.arange(300, L)
        for dst in rng.choice(pool, size=min(L // 20, len(pool)), replace=False):
            src = dst - rng.integers(100, 300)
            flat[phys[dst]] = flat[phys[src]] + 0.05 * rng.standard_normal((h_kv, d)).astype(np.float32)
    c.k_cache[0] = torch.from_numpy(Kc).to(torch.bfloat16)
    dc = DeviceCase(c)
    desc = _desc(zp, c)
    Lmax = max(lens)
    S0 = (rng.random((B, h_kv, Lmax)) / 100).astype(np.float32)
    params = zp.score_params(window=16, lightning=False)
    prm = pipeline.ScoreParams(window=16, lightning=False)
    S = torch.from_numpy(S0.copy()).cuda()
    F = torch.zeros(c.n_total, b, h_kv, device="cuda")
    first = torch.ones(B, dtype=torch.uint8, device="cuda")
    scores = torch.full((B, h_kv, Lmax), -3.0, device="cuda")
    zp.zp_score_tokens(desc, params, dc.K[0], dc.table, dc.lens, first, S, F, scores)
    k = (N_max - 1) * b
    keep = torch.empty(B, h_kv, k, dtype=torch.int32, device="cuda")
    S2 = torch.from_numpy(S0.copy()).cuda()
    targets = c.block_table[:, : N_max - 1].contiguous().cuda()
    zp.zp_compress_layers(desc, params, dc.K[0], dc.V[0], dc.table, dc.lens, first, S2, F, targets, k, keep, Lmax)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    got = scores.cpu().numpy()
    K0 = c.k_cache[0].float().numpy()
    V0 = c.v_cache[0].float().numpy()
    Kg, Vg = dc.K[0].float().cpu().numpy(), dc.V[0].float().cpu().numpy()
    kept = keep.cpu().numpy()
    swaps, fired = 0, 0
    for s, L in enumerate(lens):
        Fref = np.zeros((c.n_total, b, h_kv))
        sref = pipeline.final_scores(S0[s, :, :L].astype(np.float64), K0, Fref, c.block_table[s].numpy(), L, b,
                                     True, prm)
        fin = np.isfinite(sref)
        np.testing.assert_allclose(got[s, :, :L][fin], sref[fin], **TOL_SCORE["bf16"])
        for h in range(h_kv):
            swaps += keep_sets_match(kept[s, h], oracle.topk_keep(sref[h], k)[0], sref[h], k, L)
            for r in range(0, k, 7):
                pos = kept[s, h, r]
                sb, ss = c.block_table[s, pos // b], pos % b
                db, ds = c.block_table[s, r // b], r % b
                assert np.array_equal(Kg[db, ds, h], K0[sb, ss, h])
                assert np.array_equal(Vg[db, ds, h], V0[sb, ss, h])
        keys = pipeline.gather_rows(K0, c.block_table[s].numpy(), L, b)[:, 0].astype(np.float64)
        n = np.linalg.norm(keys, axis=1)
        cosm = (keys @ keys.T) / np.outer(n, n)
        np.fill_diagonal(cosm, 0)
        fired += int((cosm > 0.9).any(axis=0).sum())
    assert fired > 50  # the zeroing rule acted on many columns
    print("reported near-tie swaps:", swaps, "columns with a zeroed entry (head 0):", fired)


@pytest.mark.parametrize("w", [4, 8, 16])
def test_tiny_every_flag_combination(zp, w):
    """The tiny workload (4 sequences, 8q/2kv/64, fp32, b 16, N_max 4, 80-150
    tokens, near-duplicate keys) through zp_compress_layers under every
    combination of the scoring switches -- global score on/off, pooling
    never / first / every, redundancy off / lightning / all pairs, first or
    later compression -- at window w: final scores against the oracle at the
    fp32 tolerance, keep sets equal up to reported near-ties, and the moved
    key rows bitwise."""
    import itertools
    B, h_q, h_kv, d, b, N_max = 4, 8, 2, 64, 16, 4
    c = _block_aligned_case(1200 + w, B, h_q, h_kv, d, b, 80, 150, "f32", dup=True, spare=B * N_max)
    desc = _desc(zp, c)
    lens = c.seq_lens.tolist()
    Lmax = max(lens)
    k = (N_max - 1) * b
    rng = np.random.default_rng(1210 + w)
    S0 = (rng.random((B, h_kv, Lmax)) / 100).astype(np.float32)
    F0 = (rng.random((c.n_total, b, h_kv)) / 80).astype(np.float32)
    free = c.free_blocks.numpy()
    targets = torch.from_numpy(np.stack([free[i * (N_max - 1):(i + 1) * (N_max - 1)]
                                         for i in range(B)]).astype(np.int32)).cuda()
    K0 = c.k_cache[0].float().numpy()
    swaps = combos = 0
    for use_global, pool_policy, redundancy, first in itertools.product((True, False), (0, 1, 2),
                                                                        ("off", "lightning", "all"), (1, 0)):
        kw = dict(window=w, use_global=use_global, pool_policy=pool_policy,
                  use_similarity=redundancy != "off", lightning=redundancy != "all")
        params = zp.score_params(**kw)
        prm = pipeline.ScoreParams(window=w, use_global=use_global, pool_policy=pool_policy,
                                   use_similarity=redundancy != "off", lightning=redundancy != "all")
        dc = DeviceCase(c)
        S = torch.from_numpy(S0.copy()).cuda()
        F = torch.from_numpy(F0.copy()).cuda()
        fc = torch.full((B,), first, dtype=torch.uint8, device="cuda")
        scores = torch.full((B, h_kv, Lmax), -5.0, device="cuda")
        keep = torch.empty(B, h_kv, k, dtype=torch.int32, device="cuda")
        zp.zp_compress_layers(desc, params, dc.K[0], dc.V[0], dc.table, dc.lens, fc, S, F, targets, k, keep, Lmax,
                              scores_out=scores)
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        got, kept, Kg = scores.cpu().numpy(), keep.cpu().numpy(), dc.K[0].cpu().numpy()
        Fref = F0.astype(np.float64).copy()
        for s, L in enumerate(lens):
            want = pipeline.final_scores(S0[s, :, :L].astype(np.float64), K0, Fref, c.block_table[s].numpy(), L, b,
                                         bool(first), prm)
            fin = np.isfinite(want)
            assert np.array_equal(fin, np.isfinite(got[s, :, :L])), kw
            np.testing.assert_allclose(got[s, :, :L][fin], want[fin], **TOL_SCORE["f32"], err_msg=str(kw))
            for h in range(h_kv):
                swaps += keep_sets_match(kept[s, h], oracle.topk_keep(want[h], k)[0], want[h], k, L)
                tg = targets[s].cpu().numpy()
                for r, pos in enumerate(kept[s, h][:min(k, L)]):
                    src = K0[c.block_table[s, pos // b], pos % b, h]
                    assert np.array_equal(Kg[tg[r // b], r % b, h], src)
        combos += 1
    assert combos == 36
    print("w=%d combinations: %d, reported near-tie swaps: %d" % (w, combos, swaps))
