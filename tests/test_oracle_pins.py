"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks an oracle function against something the paper or plain
mathematics fixes: a library routine computing the same definition, a closed
form, an invariant, a special case, exhaustive search on tiny inputs, or the
worked example of the paper's Figure 1.  A plausible slip in the oracle (a
dropped term, a swapped index, a wrong mask or tie rule) fails at least one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import zp_inputs
from oracle import pipeline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.float().numpy()


def _case(seed, B, h_q, h_kv, d, b, lens=None, len_range=(1, 40), spare=0):
    return zp_inputs.make_paged_case(seed, B, h_q, h_kv, d, b, lens=lens, len_range=len_range,
                                     dtype="f32", spare_blocks=spare)


# --------------------------------------------------------------------------- decode attention
@pytest.mark.parametrize("h_q,h_kv,d,b", [(4, 4, 16, 4), (8, 2, 32, 8), (6, 1, 8, 16)])
def test_decode_matches_torch_sdpa(orc, h_q, h_kv, d, b):
    """Library pin: torch's scaled_dot_product_attention in fp64 on the gathered rows."""
    c = _case(11, 5, h_q, h_kv, d, b, len_range=(1, 45))
    out = orc.decode_attention(_np(c.q), _np(c.k_cache[0]), _np(c.v_cache[0]), c.block_table.numpy(),
                               c.seq_lens.numpy())
    g = h_q // h_kv
    for s in range(c.B):
        L = int(c.seq_lens[s])
        K = zp_inputs.gather_tokens(c.k_cache[0], c.block_table[s], L, b).double()  # [L][h_kv][d]
        V = zp_inputs.gather_tokens(c.v_cache[0], c.block_table[s], L, b).double()
        Kh = K.permute(1, 0, 2).repeat_interleave(g, dim=0)  # [h_q][L][d]
        Vh = V.permute(1, 0, 2).repeat_interleave(g, dim=0)
        qh = c.q[s].double().unsqueeze(1)  # [h_q][1][d]
        ref = torch.nn.functional.scaled_dot_product_attention(qh, Kh, Vh).squeeze(1)
        np.testing.assert_allclose(out[s], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_decode_single_token_returns_its_value(orc):
    c = _case(12, 3, 8, 2, 16, 4, lens=[1, 1, 1])
    out = orc.decode_attention(_np(c.q), _np(c.k_cache[0]), _np(c.v_cache[0]), c.block_table.numpy(),
                               c.seq_lens.numpy())
    for s in range(3):
        blk = int(c.block_table[s, 0])
        for h in range(8):
            np.testing.assert_array_equal(out[s, h], _np(c.v_cache[0, blk, 0, h // 4]))


def test_decode_zero_query_is_mean_of_values(orc):
    c = _case(13, 4, 4, 2, 8, 4, len_range=(3, 30))
    q = np.zeros_like(_np(c.q))
    out, probs = orc.decode_attention(q, _np(c.k_cache[0]), _np(c.v_cache[0]), c.block_table.numpy(),
                                      c.seq_lens.numpy(), want_probs=True)
    for s in range(c.B):
        L = int(c.seq_lens[s])
        V = zp_inputs.gather_tokens(c.v_cache[0], c.block_table[s], L, 4).double().numpy()
        for h in range(4):
            np.testing.assert_allclose(out[s, h], V[:, h // 2].mean(axis=0), rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(probs[s, h, :L], 1.0 / L, rtol=1e-13)


def test_decode_invariant_to_physical_block_permutation(orc):
    c = _case(14, 3, 4, 2, 8, 4, len_range=(5, 30), spare=3)
    base = orc.decode_attention(_np(c.q), _np(c.k_cache[0]), _np(c.v_cache[0]), c.block_table.numpy(),
                                c.seq_lens.numpy())
    perm = torch.randperm(c.n_total, generator=torch.Generator().manual_seed(5))
    inv = torch.argsort(perm)
    K2 = c.k_cache[0][inv]          # new block j holds old block perm[j]... relabel by inv
    V2 = c.v_cache[0][inv]
    table = c.block_table.clone()
    mask = table >= 0
    table[mask] = perm[table[mask].long()].to(torch.int32)
    out = orc.decode_attention(_np(c.q), _np(K2), _np(V2), table.numpy(), c.seq_lens.numpy())
    np.testing.assert_allclose(out, base, rtol=0, atol=0)


def test_decode_probabilities_sum_to_one(orc):
    c = _case(15, 4, 8, 4, 16, 8, len_range=(1, 50))
    _, probs = orc.decode_attention(_np(c.q), _np(c.k_cache[0]), _np(c.v_cache[0]),
                                    c.block_table.numpy(), c.seq_lens.numpy(), want_probs=True)
    for s in range(c.B):
        L = int(c.seq_lens[s])
        np.testing.assert_allclose(probs[s, :, :L].sum(axis=1), 1.0, rtol=1e-13)
        assert np.all(probs[s, :, L:] == 0)


# --------------------------------------------------------------------------- window score
def test_window_score_g1_sums_to_one(orc):
    c = _case(21, 1, 2, 2, 16, 4, lens=[37])
    qw = zp_inputs.normal((5, 2, 16), 3).numpy()
    S = orc.window_score(qw, _np(c.k_cache[0]), c.block_table[0].numpy(), 37, 5)
    np.testing.assert_allclose(S.sum(axis=1), 1.0, rtol=1e-13)


def test_window_score_group_sum_between_one_and_g(orc):
    c = _case(22, 1, 8, 2, 16, 4, lens=[29])
    qw = zp_inputs.normal((4, 8, 16), 4).numpy()
    S = orc.window_score(qw, _np(c.k_cache[0]), c.block_table[0].numpy(), 29, 4)
    tot = S.sum(axis=1)
    assert np.all(tot >= 1.0 - 1e-12) and np.all(tot <= 4.0 + 1e-12)
    assert np.all(tot > 1.0 + 1e-6)  # max over 4 random heads exceeds any single head


def test_window_score_w1_is_decode_group_max(orc):
    """w = 1: the window is the newest query alone, i.e. one decode step."""
    c = _case(23, 1, 8, 2, 16, 4, lens=[23])
    q = zp_inputs.normal((1, 8, 16), 5).numpy()
    S = orc.window_score(q, _np(c.k_cache[0]), c.block_table[0].numpy(), 23, 1)
    _, probs = orc.decode_attention(q, _np(c.k_cache[0]), _np(c.v_cache[0]), c.block_table[:1].numpy(),
                                    np.array([23], dtype=np.int32), want_probs=True)
    ref = probs[0].reshape(2, 4, 23).max(axis=1)
    np.testing.assert_allclose(S, ref, rtol=1e-13, atol=0)


def test_window_score_masks_future_tokens(orc):
    """The newest token is seen only by the last window row (causal mask)."""
    w, L = 4, 26
    c = _case(24, 1, 4, 1, 8, 4, lens=[L])
    qw = zp_inputs.normal((w, 4, 8), 6).numpy()
    S = orc.window_score(qw, _np(c.k_cache[0]), c.block_table[0].numpy(), L, w)
    _, probs = orc.decode_attention(qw[w - 1:w], _np(c.k_cache[0]), _np(c.v_cache[0]),
                                    c.block_table[:1].numpy(), np.array([L], dtype=np.int32),
                                    want_probs=True)
    np.testing.assert_allclose(S[0, L - 1], probs[0, :, L - 1].max() / w, rtol=1e-13)


def _crossed_focus_case(L, b, d, x):
    """One kv head (g = 2, w = 2) over orthonormal keys k_t = e_t, and window
    queries that put logit x on one token and 0 on every other: head 0 looks at
    token A from the first window row and at token B from the second, head 1
    the other way round.  Returns (q_window [2][2][d], k_cache, table_row, A, B)."""
    assert d >= L and L % b == 0
    nb = L // b
    K = np.zeros((nb, b, 1, d), dtype=np.float32)
    for t in range(L):
        K[t // b, t % b, 0, t] = 1.0
    A, B = 3, 7
    beta = x * math.sqrt(d)  # q . e_t / sqrt(d) = x
    qw = np.zeros((2, 2, d), dtype=np.float32)
    qw[0, 0, A] = qw[1, 1, A] = beta
    qw[0, 1, B] = qw[1, 0, B] = beta
    return qw, K, np.arange(nb, dtype=np.int32), A, B


def test_window_score_order_closed_form(orc):
    """App. C.2 takes the max over the query heads of a kv head first and the
    mean over the window rows second.  With one-hot-like attention the softmax
    is a closed form: n visible tokens, logit x on the focused one, 0 elsewhere
    give p_focus = e^x/(e^x + n - 1) and p_other = 1/(e^x + n - 1).  Row 0 sees
    n0 = L-1 tokens, row 1 sees n1 = L.  Max then mean gives, for A and B,
    (pf(n0) + pf(n1))/2; mean then max would give max of (pf(n0)+po(n1))/2 and
    (po(n0)+pf(n1))/2, which is smaller by a wide margin."""
    L, b, d, x = 12, 4, 16, 2.0
    qw, K, row, A, B = _crossed_focus_case(L, b, d, x)
    x = float(np.float32(x * math.sqrt(d))) / math.sqrt(d)  # the logit the float query gives
    pf = lambda n: math.exp(x) / (math.exp(x) + n - 1)
    po = lambda n: 1.0 / (math.exp(x) + n - 1)
    n0, n1 = L - 1, L
    S = orc.window_score(qw, K, row, L, 2)
    want_AB = (pf(n0) + pf(n1)) / 2
    swapped_AB = max((pf(n0) + po(n1)) / 2, (po(n0) + pf(n1)) / 2)
    assert want_AB - swapped_AB > 0.1
    for t in range(L):
        if t in (A, B):
            want = want_AB
        elif t == L - 1:  # seen by the second row only
            want = po(n1) / 2
        else:
            want = (po(n0) + po(n1)) / 2
        assert abs(S[0, t] - want) <= 1e-14, (t, S[0, t], want)


def test_accumulated_score_order_closed_form(orc):
    """The per-decode-step accumulation over the same two window queries (the
    two steps ending at a full block) gives the same closed form."""
    L, b, d, x = 12, 4, 16, 2.0
    w = 2
    qw, K, row, A, B = _crossed_focus_case(L, b, d, x)
    x = float(np.float32(x * math.sqrt(d))) / math.sqrt(d)
    pf = lambda n: math.exp(x) / (math.exp(x) + n - 1)
    po = lambda n: 1.0 / (math.exp(x) + n - 1)
    S = np.full((L // b, b, 1), 5.0)  # stale values must be overwritten
    table = row[None, :]
    for u in range(w):
        lens = np.array([L - w + u + 1], dtype=np.int32)
        _, probs = orc.decode_attention(qw[u:u + 1], K, K, table, lens, want_probs=True)
        orc.accumulate_window_score(probs, table, lens, 1, b, w, S)
    got = pipeline.gather_slots(S, row, L, b)[0]
    assert abs(got[A] - (pf(L - 1) + pf(L)) / 2) <= 1e-14
    assert abs(got[B] - (pf(L - 1) + pf(L)) / 2) <= 1e-14
    assert abs(got[0] - (po(L - 1) + po(L)) / 2) <= 1e-14
    assert abs(got[L - 1] - po(L) / 2) <= 1e-14


def _window_score_bruteforce(qw, Kseq, w, L, g, group_first=True):
    """Masked logits in torch fp64, softmax per row over t < L, then the two
    reductions in the order asked for.  qw [w][h_q][d], Kseq [L][h_kv][d]."""
    q = torch.from_numpy(qw).double()
    k = Kseq.double()
    h_q, d = q.shape[1], q.shape[2]
    h_kv = h_q // g
    kh = k.permute(1, 0, 2).repeat_interleave(g, dim=0)  # [h_q][L][d]
    logits = torch.einsum("uhi,hti->uht", q, kh) / math.sqrt(d)  # [w][h_q][L]
    pos = torch.arange(L)
    for u in range(w):
        logits[u, :, pos > L - w + u] = -math.inf
    P = torch.softmax(logits, dim=-1).reshape(w, h_kv, g, L)
    if group_first:
        return P.amax(dim=2).mean(dim=0)  # [h_kv][L]
    return P.mean(dim=0).amax(dim=1)


@pytest.mark.parametrize("w,g", [(4, 4), (8, 2), (16, 4)])
def test_window_score_matches_masked_bruteforce_and_not_swapped_order(orc, w, g):
    """Brute force over the explicit masked logits (max over the group, then
    mean over the window) equals the oracle, and the swapped order (mean, then
    max) is far from it, so a swap in the oracle would fail here."""
    h_kv, d, b = 2, 16, 16
    h_q = h_kv * g
    L = 3 * b + 5
    c = _case(40 + w + g, 1, h_q, h_kv, d, b, lens=[L])
    qw = (zp_inputs.normal((w, h_q, d), 50 + w) * 2.0).numpy()
    S = orc.window_score(qw, _np(c.k_cache[0]), c.block_table[0].numpy(), L, w)
    Kseq = zp_inputs.gather_tokens(c.k_cache[0], c.block_table[0], L, b)
    ref = _window_score_bruteforce(qw, Kseq, w, L, g).numpy()
    np.testing.assert_allclose(S, ref, rtol=1e-12, atol=1e-15)
    swapped = _window_score_bruteforce(qw, Kseq, w, L, g, group_first=False).numpy()
    assert np.abs(S - swapped).max() > 1e-6


@pytest.mark.parametrize("w", [4, 8])
def test_accumulated_score_matches_masked_bruteforce(orc, w):
    """The decode-time accumulation over the w steps ending at a full block
    against the same brute force."""
    h_q, h_kv, d, b = 8, 2, 16, 8
    g = h_q // h_kv
    L = 4 * b
    c = _case(60 + w, 1, h_q, h_kv, d, b, lens=[L])
    qw = (zp_inputs.normal((w, h_q, d), 70 + w) * 2.0).numpy()
    S = np.zeros((c.n_total, b, h_kv))
    for u in range(w):
        lens = np.array([L - w + u + 1], dtype=np.int32)
        _, probs = orc.decode_attention(np.ascontiguousarray(qw[u:u + 1]), _np(c.k_cache[0]),
                                        _np(c.v_cache[0]), c.block_table.numpy(), lens, want_probs=True)
        orc.accumulate_window_score(probs, c.block_table.numpy(), lens, h_kv, b, w, S)
    got = pipeline.gather_slots(S, c.block_table[0].numpy(), L, b)
    Kseq = zp_inputs.gather_tokens(c.k_cache[0], c.block_table[0], L, b)
    ref = _window_score_bruteforce(qw, Kseq, w, L, g).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)
    swapped = _window_score_bruteforce(qw, Kseq, w, L, g, group_first=False).numpy()
    assert np.abs(got - swapped).max() > 1e-6


@pytest.mark.parametrize("w,b", [(4, 4), (2, 8), (8, 8), (3, 4)])
def test_accumulated_score_equals_explicit_window(orc, w, b):
    """Per-step accumulation over the w decode steps that end at a full block
    reproduces the explicit window score of App. C.2 / Alg. 1 (invariant)."""
    h_q, h_kv, d = 6, 2, 16
    lens_final = [3 * b, 5 * b, 2 * b]
    c = _case(25 + w, 3, h_q, h_kv, d, b, lens=lens_final)
    rng = np.random.default_rng(7)
    S = rng.standard_normal((c.n_total, b, h_kv))  # stale values must be overwritten
    qw = zp_inputs.normal((3, w, h_q, d), 8 + w).numpy()
    for u in range(w):
        lens = np.array([L - w + u + 1 for L in lens_final], dtype=np.int32)
        _, probs = orc.decode_attention(np.ascontiguousarray(qw[:, u]), _np(c.k_cache[0]),
                                        _np(c.v_cache[0]), c.block_table.numpy(), lens, want_probs=True)
        orc.accumulate_window_score(probs, c.block_table.numpy(), lens, h_kv, b, w, S)
    for s, L in enumerate(lens_final):
        ref = orc.window_score(qw[s], _np(c.k_cache[0]), c.block_table[s].numpy(), L, w)
        got = pipeline.gather_slots(S, c.block_table[s].numpy(), L, b)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)


def test_accumulation_skips_non_window_steps(orc):
    b, w = 8, 2
    c = _case(26, 1, 4, 2, 8, b, lens=[13])  # position 12: 12 % 8 = 4 < b - w
    S = np.full((c.n_total, b, 2), 7.0)
    _, probs = orc.decode_attention(_np(c.q), _np(c.k_cache[0]), _np(c.v_cache[0]), c.block_table.numpy(),
                                    c.seq_lens.numpy(), want_probs=True)
    orc.accumulate_window_score(probs, c.block_table.numpy(), c.seq_lens.numpy(), 2, b, w, S)
    assert np.all(S == 7.0)


# --------------------------------------------------------------------------- global score
def test_global_score_hand_worked_example(orc):
    with open(os.path.join(GOLDEN, "global_score_two_blocks.json")) as f:
        ex = json.load(f)
    b = ex["b"]
    table = np.array([1, 0], dtype=np.int32)  # logical block 0 -> physical 1
    F = np.zeros((2, b, 1))
    Fin = np.array(ex["F_in"])
    F[1, :, 0] = Fin[:2]
    F[0, :, 0] = Fin[2:]
    S = np.array([ex["S_in"]], dtype=np.float64)
    orc.global_score(S, F, table, b, first=False, alpha=ex["alpha"])
    np.testing.assert_allclose(S[0], ex["S_out"], rtol=1e-15)
    np.testing.assert_allclose(np.concatenate([F[1, :, 0], F[0, :, 0]]), ex["F_out"], rtol=1e-15)


def test_global_score_first_compression_copies(orc):
    rng = np.random.default_rng(3)
    b, h_kv, L = 4, 3, 14
    table = np.array([5, 2, 7, 0], dtype=np.int32)
    F = rng.standard_normal((8, b, h_kv))
    S = rng.random((h_kv, L))
    S0 = S.copy()
    orc.global_score(S, F, table, b, first=True, alpha=0.8)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_array_equal(pipeline.gather_slots(F, table, L, b), S0)


def test_global_score_alpha_zero_is_identity_on_nonnegative(orc):
    rng = np.random.default_rng(4)
    b, h_kv, L = 4, 2, 16
    table = np.array([3, 1, 0, 2], dtype=np.int32)
    F = rng.random((4, b, h_kv)) * 5
    S = rng.random((h_kv, L))
    S0 = S.copy()
    orc.global_score(S, F, table, b, first=False, alpha=0.0)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_array_equal(pipeline.gather_slots(F, table, L, b), S0)


# --------------------------------------------------------------------------- pooling
@pytest.mark.parametrize("kernel", [1, 3, 5, 7, 9])
def test_max_pool_matches_torch(orc, kernel):
    x = np.random.default_rng(kernel).standard_normal(57)
    y = orc.max_pool(x, kernel)
    ref = torch.nn.functional.max_pool1d(torch.from_numpy(x)[None, None], kernel, stride=1,
                                         padding=kernel // 2)[0, 0].numpy()
    np.testing.assert_array_equal(y, ref)


def test_max_pool_kernel_one_is_identity_and_monotone_shift(orc):
    x = np.arange(20, dtype=np.float64)
    np.testing.assert_array_equal(orc.max_pool(x, 1), x)
    np.testing.assert_array_equal(orc.max_pool(x, 7), np.minimum(x + 3, 19))


# --------------------------------------------------------------------------- redundancy
def _softmax(z):
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


@pytest.mark.parametrize("lightning", [0, 1])
def test_redundancy_orthogonal_keys_uniform(orc, lightning):
    L, d = 12, 16
    keys = np.eye(d, dtype=np.float32)[:L] * 3.0
    R = orc.redundancy(keys, 4, 0.9, 0.4, lightning)
    np.testing.assert_allclose(R, 1.0 / L, rtol=1e-14)


@pytest.mark.parametrize("m", [2, 3, 8])
def test_redundancy_identical_keys_closed_form(orc, m):
    """One block of m identical keys: rho[m-1] = 0, rho[m-2] = m-2, others m-1."""
    d, tau = 8, 0.4
    keys = np.tile(np.arange(1, d + 1, dtype=np.float32), (m, 1))
    rho = np.full(m, m - 1.0)
    rho[m - 1] = 0.0
    rho[m - 2] = m - 2.0
    ref = _softmax(rho / (m * tau))
    for lightning in (0, 1):
        R = orc.redundancy(keys, 8, 0.9, tau, lightning)
        np.testing.assert_allclose(R, ref, rtol=1e-12)


def test_redundancy_lightning_blocks_closed_form(orc):
    """Lightning with b = 4 on 10 identical keys: the pattern repeats per block,
    the partial last block (2 keys) follows the same rule with m = 2."""
    b, L, tau = 4, 10, 0.4
    keys = np.tile(np.array([1, -2, 3, 0.5], dtype=np.float32), (L, 1))
    rho = []
    for m in (4, 4, 2):
        r = np.full(m, m - 1.0)
        r[m - 1] = 0.0
        r[m - 2] = m - 2.0
        rho.append(r)
    ref = _softmax(np.concatenate(rho) / (L * tau))
    np.testing.assert_allclose(orc.redundancy(keys, b, 0.9, tau, 1), ref, rtol=1e-12)


def test_redundancy_lightning_equals_full_when_blocks_orthogonal(orc):
    """If keys of different blocks are orthogonal, the full (all-pairs) score and
    the same-block lightning score coincide."""
    rng = np.random.default_rng(9)
    b, nblk, d = 4, 3, 12
    keys = np.zeros((b * nblk, d), dtype=np.float32)
    for i in range(nblk):
        base = rng.standard_normal(4)
        for j in range(b):
            keys[i * b + j, 4 * i:4 * i + 4] = base + 0.1 * rng.standard_normal(4)
    full = orc.redundancy(keys, b, 0.9, 0.4, 0)
    light = orc.redundancy(keys, b, 0.9, 0.4, 1)
    np.testing.assert_allclose(light, full, rtol=1e-14)
    assert np.ptp(full) > 1e-3  # non-trivial: some pairs above the threshold


@pytest.mark.parametrize("lightning", [0, 1])
def test_redundancy_brute_force_with_duplicates(orc, lightning):
    """Pure-Python brute force over the L x L pair matrix with the domain mask
    (same block for lightning), keys with planted near-duplicates so the
    threshold rule fires, a ragged last block."""
    rng = np.random.default_rng(17 + lightning)
    L, b, d, p, tau = 23, 8, 6, 0.5, 0.4
    keys = rng.standard_normal((L, d)).astype(np.float32)
    for t in (3, 5, 9, 12, 13, 20, 22):
        keys[t] = keys[t - 1 - (t % 2)] + 0.05 * rng.standard_normal(d).astype(np.float32)
    k = keys.astype(np.float64)
    C = [[0.0] * L for _ in range(L)]
    for r in range(L):
        for c in range(L):
            if r != c and (not lightning or r // b == c // b):
                C[r][c] = sum(k[r, i] * k[c, i] for i in range(d)) / (
                    np.sqrt(sum(x * x for x in k[r])) * np.sqrt(sum(x * x for x in k[c])))
    fired = 0
    for c in range(L):
        above = [r for r in range(L) if C[r][c] > p]
        if above:
            C[max(above)][c] = 0.0
            fired += 1
    rho = [sum(C[r]) / (L * tau) for r in range(L)]
    np.testing.assert_allclose(orc.redundancy(keys, b, p, tau, lightning), _softmax(rho), rtol=1e-12)
    assert fired >= 6


@pytest.mark.parametrize("m", [2, 5, 9])
def test_redundancy_rho_identical_keys_closed_form(orc, m):
    """All-pairs row sums of m identical keys: rho[m-1] = 0, rho[m-2] = m-2,
    others m-1, from the full function and row by row."""
    keys = np.tile(np.array([2, -1, 0.5, 3], dtype=np.float32), (m, 1))
    want = np.full(m, m - 1.0)
    want[m - 1] = 0.0
    want[m - 2] = m - 2.0
    np.testing.assert_allclose(orc.redundancy_rho(keys, m, 0.9, 0), want, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(orc.redundancy_rho_rows(keys, 0.9, np.arange(m)), want, rtol=1e-13, atol=1e-13)


def test_redundancy_rho_orthogonal_keys_zero(orc):
    keys = np.eye(10, dtype=np.float32)[:7] * 2.5
    np.testing.assert_array_equal(orc.redundancy_rho(keys, 4, 0.9, 0), np.zeros(7))
    np.testing.assert_array_equal(orc.redundancy_rho_rows(keys, 0.9, [0, 3, 6]), np.zeros(3))


@pytest.mark.parametrize("p", [0.5, -0.3])
def test_redundancy_rho_brute_force(orc, p):
    """Pure-Python brute force of the all-pairs row sums (zero diagonal, the
    newest row above p zeroed in every column, zero-norm key included), for the
    full function and the selected-rows function; with p < 0 the zeroed
    diagonal itself can be a column's newest entry above p."""
    rng = np.random.default_rng(31)
    L, d = 29, 5
    keys = rng.standard_normal((L, d)).astype(np.float32)
    for t in (4, 7, 11, 15, 16, 22, 27, 28):
        keys[t] = keys[t - 3 - (t % 4)] + 0.05 * rng.standard_normal(d).astype(np.float32)
    keys[9] = 0.0
    k = keys.astype(np.float64)
    nrm = [np.sqrt(sum(x * x for x in k[r])) for r in range(L)]
    C = [[0.0] * L for _ in range(L)]
    for r in range(L):
        for c in range(L):
            if r != c and nrm[r] > 0 and nrm[c] > 0:
                C[r][c] = sum(k[r, i] * k[c, i] for i in range(d)) / (nrm[r] * nrm[c])
    for c in range(L):
        above = [r for r in range(L) if C[r][c] > p]
        if above:
            C[max(above)][c] = 0.0
    want = np.array([sum(C[r]) for r in range(L)])
    np.testing.assert_allclose(orc.redundancy_rho(keys, 4, p, 0), want, rtol=1e-12, atol=1e-12)
    rows = np.array([0, 3, 9, 11, 16, 27, 28], dtype=np.int32)
    np.testing.assert_allclose(orc.redundancy_rho_rows(keys, p, rows), want[rows], rtol=1e-12, atol=1e-12)
    tau = 0.3
    np.testing.assert_allclose(orc.redundancy(keys, 4, p, tau, 0), _softmax(want / (L * tau)), rtol=1e-12)


@pytest.mark.parametrize("p", [-2.0, -1.5])
def test_redundancy_rho_lightning_below_minus_one_closed_form(orc, p):
    """Lightning row sums (App. C.5, same-block pairs of C.7) with p < -1:
    every cosine, and every column's zeroed diagonal, exceeds p, so in each
    column the newest row of the block loses its entry.  Per block -- the last
    one partial -- the block's last row sums to 0 and every other row to its
    cosines with the block's other tokens; a zero key adds nothing.  Taking
    the diagonal out of the newest-row search, letting rows of another block
    (or past the sequence's end) take part, or keeping the zeroed entry would
    each change some row."""
    rng = np.random.default_rng(44)
    L, b, d = 27, 8, 5  # blocks of 8, 8, 8 and one of 3
    keys = rng.standard_normal((L, d)).astype(np.float32)
    keys[10] = 0.0
    k = keys.astype(np.float64)
    nrm = [float(np.sqrt(sum(x * x for x in k[r]))) for r in range(L)]
    want = np.zeros(L)
    for b0 in range(0, L, b):
        blk = list(range(b0, min(L, b0 + b)))
        for r in blk[:-1]:
            for c in blk:
                if c != r and nrm[r] > 0 and nrm[c] > 0:
                    want[r] += sum(k[r, i] * k[c, i] for i in range(d)) / (nrm[r] * nrm[c])
    np.testing.assert_allclose(orc.redundancy_rho(keys, b, p, 1), want, rtol=1e-12, atol=1e-12)


def test_redundancy_zero_norm_key_has_no_similarity(orc):
    keys = np.array([[0, 0], [1, 0], [0, 1]], dtype=np.float32)
    R = orc.redundancy(keys, 4, 0.5, 1.0, 0)
    np.testing.assert_allclose(R, 1.0 / 3, rtol=1e-14)


def test_redundancy_threshold_zeroes_newest_similar(orc):
    """Two near-duplicate keys and one unrelated key: the column of the older
    duplicate loses its entry at the newer one, so the newer one is less
    redundant (C.5: newer tokens are retained)."""
    keys = np.array([[1, 0, 0], [0, 0, 1], [1, 0.01, 0]], dtype=np.float32)
    tau = 0.5
    R = orc.redundancy(keys, 4, 0.9, tau, 0)
    c = float(np.dot(keys[0], keys[2]) / np.linalg.norm(keys[0]) / np.linalg.norm(keys[2]))
    # column 0: last row > p is row 2 -> zeroed; column 2: last row > p is row 0 -> zeroed
    rho = np.array([0.0, 0.0, 0.0]) / (3 * tau)
    np.testing.assert_allclose(R, _softmax(rho), rtol=1e-14)
    keys3 = np.array([[1, 0, 0], [1, 0.02, 0], [1, 0.01, 0]], dtype=np.float32)
    R3 = orc.redundancy(keys3, 4, 0.9, tau, 0)
    # every column keeps exactly one off-diagonal entry; row sums by hand:
    k64 = keys3.astype(np.float64)
    n = np.linalg.norm(k64, axis=1)
    C = (k64 @ k64.T) / np.outer(n, n)
    np.fill_diagonal(C, 0)
    C[2, 0] = 0  # column 0: rows 1, 2 above p, newest is 2
    C[2, 1] = 0  # column 1: rows 0, 2 above p, newest is 2
    C[1, 2] = 0  # column 2: rows 0, 1 above p, newest is 1
    np.testing.assert_allclose(R3, _softmax(C.sum(axis=1) / (3 * tau)), rtol=1e-13)
    assert c > 0.9


def test_combine_lambda_zero_and_window(orc):
    S = np.random.default_rng(1).random(10)
    R = np.random.default_rng(2).random(10)
    out = orc.combine_and_window(S, 3, 0.0, R)
    np.testing.assert_array_equal(out[:7], S[:7])
    assert np.all(np.isinf(out[7:])) and np.all(out[7:] > 0)
    out2 = orc.combine_and_window(S, 0, 0.5, R)
    np.testing.assert_allclose(out2, S - 0.5 * R, rtol=1e-15)


def test_combine_hand_worked_example(orc):
    """Eq. (4) with the window of App. C.6, worked by hand: S - lambda R on the
    first L - w tokens, +inf on the last w (binary fractions, so exact)."""
    S = np.array([0.5, 0.25, 0.875, 0.125, 0.75])
    R = np.array([0.25, 0.5, 0.125, 0.0625, 0.0625])
    out = orc.combine_and_window(S, 2, 2.0, R)
    np.testing.assert_array_equal(out[:3], [0.0, -0.75, 0.625])
    assert np.all(np.isposinf(out[3:]))


# --------------------------------------------------------------------------- top-k
def _dominates(s, a, c):
    return s[a] > s[c] or (s[a] == s[c] and a > c)


@pytest.mark.parametrize("seed", range(6))
def test_topk_exhaustive(orc, seed):
    """Exhaustive search: the kept set is the one subset of size k every member
    of which outranks every non-member; with distinct scores it also has the
    largest score sum."""
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 11))
    k = int(rng.integers(0, L + 2))
    s = rng.integers(0, 4, size=L).astype(np.float64) if seed % 2 else rng.random(L)
    keep, tag, n = orc.topk_keep(s, k)
    if L <= k:
        assert list(keep[:L]) == list(range(L)) and np.all(keep[L:] == -1) and n == L
        return
    winners = [S for S in itertools.combinations(range(L), k)
               if all(_dominates(s, a, c) for a in S for c in set(range(L)) - set(S))]
    assert len(winners) == 1
    assert list(keep) == list(winners[0])
    assert tag.sum() == k
    if seed % 2 == 0:
        best = max(itertools.combinations(range(L), k), key=lambda S: s[list(S)].sum())
        assert list(keep) == list(best)


def test_topk_ties_prefer_newer(orc):
    keep, _, _ = orc.topk_keep(np.ones(6), 2)
    assert list(keep) == [4, 5]


def test_fig1_keep_set_and_window(orc):
    with open(os.path.join(GOLDEN, "fig1_compression.json")) as f:
        ex = json.load(f)
    N_max, b, w = ex["N_max"], ex["b"], ex["w"]
    L = len(ex["tokens"])
    k = (N_max - 1) * b
    rng = np.random.default_rng(0)
    s = rng.random(L) + 1.0
    for tok in ex["evicted"]:
        s[tok - 1] = rng.random() * 0.5
    s[14] = 0.0  # the window must survive even the lowest score
    final = orc.combine_and_window(s, w, 0.0, None)
    keep, _, n = orc.topk_keep(final, k)
    assert n == k == 12
    assert [int(t) + 1 for t in keep] == sum(ex["kept_after"], [])


# --------------------------------------------------------------------------- compaction
def test_fig1_compaction_layout(orc):
    with open(os.path.join(GOLDEN, "fig1_compression.json")) as f:
        ex = json.load(f)
    b = ex["b"]
    h_kv, d = 1, 3
    phys = {"a": 2, "b": 0, "c": 5, "d": 3}
    cache = np.zeros((6, b, h_kv, d), dtype=np.float32)
    table = [phys[x] for x in ex["blocks_before"]]
    for t, tok in enumerate(ex["tokens"]):
        cache[table[t // b], t % b, 0, :] = tok
    tag = np.ones(16, dtype=np.uint8)
    for tok in ex["evicted"]:
        tag[tok - 1] = 0
    moved = orc.compact_alg4(cache, d * 4, b, h_kv, 0, table, table, tag)
    assert moved == 12
    for i, row in enumerate(ex["kept_after"]):
        blk = phys[ex["blocks_after"][i]]
        assert list(cache[blk, :, 0, 0]) == row
        assert np.all(cache[blk, :, 0, :] == np.array(row, dtype=np.float32)[:, None])


def test_compaction_out_of_place_matches_in_place_and_is_bitwise(orc):
    rng = np.random.default_rng(5)
    b, h_kv, d, N = 4, 2, 8, 5
    raw = rng.integers(0, 2 ** 16, size=(12, b, h_kv, d), dtype=np.uint16)  # any bit pattern
    src = np.array([7, 1, 9, 4, 0], dtype=np.int32)
    dst = np.array([2, 3, 10, 11], dtype=np.int32)
    L = 19
    for kvh in range(h_kv):
        tag = np.zeros(L, dtype=np.uint8)
        tag[np.sort(rng.choice(L, 12, replace=False))] = 1
        a = raw.copy()
        bb = raw.copy()
        orc.compact_alg4(a, d * 2, b, h_kv, kvh, src, src, tag)
        orc.compact_alg4(bb, d * 2, b, h_kv, kvh, src, dst, tag)
        kept = np.nonzero(tag)[0]
        for r, pos in enumerate(kept):
            want = raw[src[pos // b], pos % b, kvh]
            assert np.array_equal(a[src[r // b], r % b, kvh], want)
            assert np.array_equal(bb[dst[r // b], r % b, kvh], want)
        np.testing.assert_array_equal(bb[src][:, :, kvh], raw[src][:, :, kvh])  # sources untouched
        other = 1 - kvh
        np.testing.assert_array_equal(a[:, :, other], raw[:, :, other])


# --------------------------------------------------------------------------- trigger + planner
def test_fig1_trigger(orc):
    assert orc.needs_compression(16, 4, 4)
    assert not orc.needs_compression(15, 4, 4)
    assert not orc.needs_compression(12, 4, 4)
    assert orc.needs_compression(20, 4, 4)  # prefill beyond N_max blocks
    assert not orc.needs_compression(0, 4, 4)


def test_fig1_plan_no_sharing(orc):
    ref = np.zeros(10, dtype=np.int32)
    table = np.array([2, 0, 5, 3], dtype=np.int32)  # a, b, c, d
    ref[table] = 1
    plan = orc.plan_targets(table, 4, ref, np.array([], dtype=np.int32))
    assert list(plan["targets"]) == [2, 0, 5]
    assert list(plan["new_table"]) == [2, 0, 5, 3]
    assert len(plan["released"]) == 0 and plan["fresh_used"] == 0


def test_plan_prefill_beyond_budget_releases_tail(orc):
    ref = np.zeros(10, dtype=np.int32)
    table = np.array([2, 0, 5, 3, 8, 9], dtype=np.int32)
    ref[table] = 1
    plan = orc.plan_targets(table, 4, ref, np.array([], dtype=np.int32))
    assert list(plan["new_table"]) == [2, 0, 5, 3]
    assert sorted(plan["released"]) == [8, 9]


def test_plan_shared_prefix_at_least_budget(orc):
    """N_prefix >= N_max - 1: N_max - 1 new target blocks (§4.4, first case)."""
    N_max = 4
    ref = np.zeros(20, dtype=np.int32)
    table = np.array([0, 1, 2, 3, 4, 5], dtype=np.int32)
    ref[table] = 1
    ref[[0, 1, 2, 3]] = 3  # four shared prefix blocks
    plan = orc.plan_targets(table, N_max, ref, np.array([10, 11, 12, 13, 14], dtype=np.int32))
    assert list(plan["targets"]) == [10, 11, 12]
    assert list(plan["new_table"]) == [10, 11, 12, 13]  # reserved must not be shared
    assert sorted(plan["released"]) == [4, 5]
    assert sorted(plan["dropped_shared"]) == [0, 1, 2, 3]
    assert plan["fresh_used"] == 4


def test_plan_shared_prefix_below_budget(orc):
    """N_prefix < N_max - 1: N_prefix new blocks + own blocks (§4.4, second case)."""
    N_max = 5
    ref = np.zeros(20, dtype=np.int32)
    table = np.array([0, 1, 2, 3, 4, 5, 6], dtype=np.int32)
    ref[table] = 1
    ref[[0, 1]] = 2
    plan = orc.plan_targets(table, N_max, ref, np.array([15, 16, 17], dtype=np.int32))
    assert list(plan["targets"]) == [15, 16, 2, 3]
    assert list(plan["new_table"]) == [15, 16, 2, 3, 4]
    assert sorted(plan["released"]) == [5, 6]
    assert sorted(plan["dropped_shared"]) == [0, 1]
    assert plan["fresh_used"] == 2
    # conservation: every old block is kept, released or left (shared)
    kept_own = set(plan["new_table"]) & set(table.tolist())
    assert kept_own | set(plan["released"]) | set(plan["dropped_shared"]) == set(table.tolist())


def test_final_scores_step_order_hand_worked(orc):
    """One sequence, one kv head, b = 2, L = 6, a later compression that pools
    (kernel 3, every compression), alpha 0.5, lambda 0.6, window 1 and
    orthogonal keys (rho = 0, so R = 1/6 for every token).  In the pages'
    order -- the global score (Alg. 2: max(alpha F, S) before the last block),
    max pooling of it (eq. 3), S - lambda R (eq. 4), the window (C.6) -- the
    scores are [0.3, 0.3, 0.2, 0.2, 0.5, +inf], worked by hand; pooling before
    the global score would give 0.2 at token 1."""
    b, L = 2, 6
    S = np.array([[0.1, 0.2, 0.3, 0.1, 0.05, 0.6]])
    F = np.zeros((3, b, 1))
    F[0, 0, 0] = 0.8
    keys = np.zeros((3, b, 1, 8), dtype=np.float32)  # [N_total][b][h_kv][d], one-hot
    for t in range(L):
        keys[t // b, t % b, 0, t] = 1.0
    prm = pipeline.ScoreParams(window=1, alpha=0.5, lam=0.6, pool_kernel=3, pool_policy=2)
    out = pipeline.final_scores(S, keys, F, np.arange(3), L, b, False, prm)
    np.testing.assert_allclose(out[0, :5], [0.3, 0.3, 0.2, 0.2, 0.5], rtol=1e-12)
    assert np.isposinf(out[0, 5])


def test_pipeline_under_budget_keeps_everything(orc):
    """A sequence at or below the budget k evicts nothing (invariant)."""
    prm = pipeline.ScoreParams(window=2, pool_kernel=3)
    c = _case(31, 1, 4, 2, 8, 4, lens=[10])
    F = np.zeros((c.n_total, 4, 2))
    S = np.random.default_rng(3).random((2, 10))
    sc = pipeline.final_scores(S, _np(c.k_cache[0]), F, c.block_table[0].numpy(), 10, 4, True, prm)
    keep = pipeline.keep_sets(sc, 12)
    assert np.all(keep[:, :10] == np.arange(10)) and np.all(keep[:, 10:] == -1)
