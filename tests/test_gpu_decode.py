"""GPU parity: append + paged decode attention + fused window score vs the oracle.

Cases span several stream-K ranges and ragged tails: tiny fp32 (the 4-sequence
parity workload), Qwen3-8B-shaped bf16 layers at reduced and full size (the
64-sequence, 1k-4k context workload, checked on sampled sequences), one long
sequence split across every CTA, many short sequences per CTA, L = 1, B = 0.
"""
import numpy as np
import pytest
import torch

import oracle
import zp_inputs
from tests.gpu_util import TOL_OUT, TOL_SCORE, DeviceCase, gather_slots

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zp():
    import compressed_paged_kv_zp_gb300 as m
    return m


def _desc(zp, c):
    return zp.cache_desc(c.h_q, c.h_kv, c.d, c.b, c.n_total,
                         torch.bfloat16 if c.dtype == "bf16" else torch.float32)


def _run_decode(zp, dc, score=None, window=0, seqs=None):
    c = dc.c
    out = torch.empty_like(dc.q)
    zp.zp_paged_decode_attn(_desc(zp, c), dc.q, dc.K[0], dc.V[0], dc.table, dc.lens, out,
                            score_accum=score, window=window)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    return out.float().cpu().numpy()


def _check_out(got, c, K, V, seqs):
    q = c.q.float().numpy()
    ref = oracle.decode_attention(q[seqs], K, V, c.block_table.numpy()[seqs], c.seq_lens.numpy()[seqs])
    np.testing.assert_allclose(got[seqs], ref, **TOL_OUT[c.dtype])
    return np.abs(got[seqs] - ref).max()


CASES = [
    # name, B, h_q, h_kv, d, b, len_range, dtype
    ("tiny_f32", 4, 8, 2, 64, 16, (80, 150), "f32"),
    ("qwen_small_bf16", 8, 32, 8, 128, 16, (1, 700), "bf16"),
    ("qwen_ragged_bf16", 37, 32, 8, 128, 16, (1, 90), "bf16"),
    ("g8_bf16", 6, 64, 8, 128, 16, (1, 300), "bf16"),
    ("d64_bf16", 5, 16, 4, 64, 32, (1, 400), "bf16"),
    ("qwen_f32", 4, 32, 8, 128, 16, (100, 400), "f32"),
]


@pytest.mark.parametrize("name,B,h_q,h_kv,d,b,lr,dtype", CASES)
def test_decode_matches_oracle(zp, name, B, h_q, h_kv, d, b, lr, dtype):
    seed = 100 + [x[0] for x in CASES].index(name)
    c = zp_inputs.make_paged_case(seed, B, h_q, h_kv, d, b, len_range=lr, dtype=dtype,
                                  spare_blocks=3)
    dc = DeviceCase(c)
    got = _run_decode(zp, dc)
    _check_out(got, c, dc.np_k(), dc.np_v(), list(range(B)))


def test_decode_edge_lengths(zp):
    lens = [1, 15, 16, 17, 31, 32, 33, 1, 2]
    c = zp_inputs.make_paged_case(5, len(lens), 32, 8, 128, 16, lens=lens, dtype="bf16")
    dc = DeviceCase(c)
    got = _run_decode(zp, dc)
    _check_out(got, c, dc.np_k(), dc.np_v(), list(range(len(lens))))


def test_decode_one_long_sequence_split_across_all_ctas(zp):
    c = zp_inputs.make_paged_case(6, 1, 32, 8, 128, 16, lens=[8190], dtype="bf16")
    dc = DeviceCase(c)
    got = _run_decode(zp, dc)
    _check_out(got, c, dc.np_k(), dc.np_v(), [0])


def test_decode_many_short_sequences(zp):
    c = zp_inputs.make_paged_case(7, 700, 32, 8, 128, 16, len_range=(1, 40), dtype="bf16")
    dc = DeviceCase(c)
    got = _run_decode(zp, dc)
    _check_out(got, c, dc.np_k(), dc.np_v(), list(range(0, 700, 7)))


def test_decode_empty_batch(zp):
    c = zp_inputs.make_paged_case(8, 1, 32, 8, 128, 16, lens=[5], dtype="bf16")
    dc = DeviceCase(c)
    out = torch.zeros(0, 32, 128, dtype=torch.bfloat16, device="cuda")
    zp.zp_paged_decode_attn(_desc(zp, c), dc.q[:0], dc.K[0], dc.V[0], dc.table[:0], dc.lens[:0], out)
    torch.cuda.synchronize()


def test_decode_full_size_qwen_layer_sampled(zp):
    """The 64-sequence, ctx 1k-4k, 32q/8kv/128 bf16 layer, at full size; outputs
    of every sequence are checked against sampled oracle sequences plus the
    window score of the same sampled sequences."""
    c = zp_inputs.make_paged_case(1002, 64, 32, 8, 128, 16, len_range=(1024, 4096), dtype="bf16")
    dc = DeviceCase(c)
    S = torch.zeros(64, 8, c.block_table.shape[1] * 16, dtype=torch.float32, device="cuda")
    got = _run_decode(zp, dc, score=S, window=16)
    seqs = [0, 9, 17, 33, 47, 63]
    K, V = dc.np_k(), dc.np_v()
    _check_out(got, c, K, V, seqs)
    ref_out, probs = oracle.decode_attention(c.q.float().numpy()[seqs], K, V, c.block_table.numpy()[seqs],
                                             c.seq_lens.numpy()[seqs], want_probs=True)
    S_ref = np.zeros((c.n_total, 16, 8))
    oracle.accumulate_window_score(probs, c.block_table.numpy()[seqs], c.seq_lens.numpy()[seqs], 8,
                                   16, 16, S_ref)
    Sg = S.cpu().numpy().astype(np.float64)
    for i, s in enumerate(seqs):
        L = int(c.seq_lens[s])
        np.testing.assert_allclose(Sg[s, :, :L], gather_slots(S_ref, c.block_table[s].numpy(), L, 16),
                                   **TOL_SCORE["bf16"])


@pytest.mark.parametrize("dtype,h_q,h_kv,d,w", [("f32", 8, 2, 64, 4), ("f32", 8, 2, 64, 16),
                                                ("bf16", 32, 8, 128, 8), ("bf16", 32, 8, 128, 16)])
def test_window_score_accumulates_over_decode_steps(zp, dtype, h_q, h_kv, d, w):
    """w decode steps with appends end at a full block; the accumulated S must
    equal the oracle's per-step accumulation and its explicit window score
    (App. C.2).  S starts with stale values that the first window row must
    overwrite."""
    b = 16
    final = [5 * b, 3 * b, 9 * b, 2 * b]
    B = len(final)
    c = zp_inputs.make_paged_case(40 + w, B, h_q, h_kv, d, b, lens=final, dtype=dtype)
    dc = DeviceCase(c)
    desc = _desc(zp, c)
    stride = c.block_table.shape[1]
    S = torch.randn(B, h_kv, stride * b, device="cuda").abs()  # stale values: overwritten at the first row
    S0 = S.cpu().numpy().astype(np.float64)
    S_ref = np.zeros((c.n_total, b, h_kv))  # the oracle's paged copy of the same rows
    for s, L in enumerate(final):
        t = np.arange(L)
        S_ref[c.block_table[s].numpy()[t // b], t % b] = S0[s, :, :L].T
    qw = zp_inputs.normal((B, w, h_q, d), 77, dtype)
    kw = zp_inputs.normal((B, w, h_kv, d), 78, dtype)
    vw = zp_inputs.normal((B, w, h_kv, d), 79, dtype)
    for u in range(w):
        lens = torch.tensor([L - w + u + 1 for L in final], dtype=torch.int32)
        lens_d = lens.cuda()
        zp.zp_append_kv(desc, kw[:, u].contiguous().cuda(), vw[:, u].contiguous().cuda(), dc.K[0],
                        dc.V[0], dc.table, lens_d)
        q = qw[:, u].contiguous().cuda()
        out = torch.empty_like(q)
        zp.zp_paged_decode_attn(desc, q, dc.K[0], dc.V[0], dc.table, lens_d, out, score_accum=S, window=w)
        torch.cuda.synchronize()
        K, V = dc.np_k(), dc.np_v()
        ref, probs = oracle.decode_attention(qw[:, u].float().numpy(), K, V, c.block_table.numpy(),
                                             lens.numpy(), want_probs=True)
        np.testing.assert_allclose(out.float().cpu().numpy(), ref, **TOL_OUT[dtype])
        oracle.accumulate_window_score(probs, c.block_table.numpy(), lens.numpy(), h_kv, b, w, S_ref)
    assert zp.zp_device_status() == (0, 0)
    Sg = S.cpu().numpy().astype(np.float64)
    K = dc.np_k()
    for s, L in enumerate(final):
        got = Sg[s, :, :L]
        np.testing.assert_allclose(got, gather_slots(S_ref, c.block_table[s].numpy(), L, b),
                                   **TOL_SCORE[dtype])
        explicit = oracle.window_score(qw[s].float().numpy(), K, c.block_table[s].numpy(), L, w)
        np.testing.assert_allclose(got, explicit, **TOL_SCORE[dtype])


@pytest.mark.parametrize("dtype,h_q,h_kv,d", [("f32", 8, 2, 64), ("bf16", 32, 8, 128)])
def test_slot_map_follows_the_request(zp, dtype, h_q, h_kv, d):
    """Query slots [§4.2, §4.3]: with a slot map, batch entry i scores into
    row score_rows[i] of S.  The batch order changes at every one of the w
    window steps (as a scheduler's running batch does) while each request
    keeps its slot; one request holds no slot (-1).  Each slot row must equal
    the oracle's accumulation for its request, the slotless request and the
    unused rows stay untouched, and the outputs match the oracle."""
    b, w = 16, 16
    final = [5 * b, 3 * b, 9 * b, 2 * b, 4 * b]
    B = len(final)
    slot = [3, 0, 5, 1, -1]  # the last request decodes without a query slot
    R = 7
    c = zp_inputs.make_paged_case(60, B, h_q, h_kv, d, b, lens=final, dtype=dtype)
    dc = DeviceCase(c)
    desc = _desc(zp, c)
    stride = c.block_table.shape[1]
    S = torch.randn(R, h_kv, stride * b, device="cuda").abs()
    S0 = S.cpu().numpy().astype(np.float64)
    S_ref = np.zeros((c.n_total, b, h_kv))
    for s, L in enumerate(final):
        if slot[s] >= 0:
            t = np.arange(L)
            S_ref[c.block_table[s].numpy()[t // b], t % b] = S0[slot[s], :, :L].T
    qw = zp_inputs.normal((B, w, h_q, d), 87, dtype)
    kw = zp_inputs.normal((B, w, h_kv, d), 88, dtype)
    vw = zp_inputs.normal((B, w, h_kv, d), 89, dtype)
    rng = np.random.default_rng(90)
    for u in range(w):
        order = rng.permutation(B)
        lens = np.array([final[s] - w + u + 1 for s in range(B)], dtype=np.int32)
        lens_d = torch.from_numpy(lens[order]).cuda()
        table_d = dc.table[torch.from_numpy(order).cuda()].contiguous()
        rows_d = torch.tensor([slot[s] for s in order], dtype=torch.int32, device="cuda")
        zp.zp_append_kv(desc, kw[order, u].contiguous().cuda(), vw[order, u].contiguous().cuda(), dc.K[0],
                        dc.V[0], table_d, lens_d)
        q = qw[order, u].contiguous().cuda()
        out = torch.empty_like(q)
        zp.zp_paged_decode_attn(desc, q, dc.K[0], dc.V[0], table_d, lens_d, out, score_accum=S, window=w,
                                score_rows=rows_d)
        torch.cuda.synchronize()
        K, V = dc.np_k(), dc.np_v()
        ref, probs = oracle.decode_attention(qw[:, u].float().numpy(), K, V, c.block_table.numpy(), lens,
                                             want_probs=True)
        got = np.empty_like(ref)
        got[order] = out.float().cpu().numpy()
        np.testing.assert_allclose(got, ref, **TOL_OUT[dtype])
        sl = [s for s in range(B) if slot[s] >= 0]
        oracle.accumulate_window_score(probs[sl], c.block_table.numpy()[sl], lens[sl], h_kv, b, w,
                                       S_ref)
    assert zp.zp_device_status() == (0, 0)
    Sg = S.cpu().numpy().astype(np.float64)
    for s, L in enumerate(final):
        if slot[s] >= 0:
            np.testing.assert_allclose(Sg[slot[s], :, :L], gather_slots(S_ref, c.block_table[s].numpy(), L, b),
                                       **TOL_SCORE[dtype])
    for r in set(range(R)) - set(slot):
        assert np.array_equal(Sg[r], S0[r])


def test_append_writes_only_the_new_slot(zp):
    c = zp_inputs.make_paged_case(9, 5, 32, 8, 128, 16, len_range=(1, 100), dtype="bf16")
    dc = DeviceCase(c)
    K0 = dc.K[0].clone()
    kn = zp_inputs.normal((5, 8, 128), 10, "bf16").cuda()
    vn = zp_inputs.normal((5, 8, 128), 11, "bf16").cuda()
    zp.zp_append_kv(_desc(zp, c), kn, vn, dc.K[0], dc.V[0], dc.table, dc.lens)
    torch.cuda.synchronize()
    expect = K0.clone()
    for s in range(5):
        P = int(c.seq_lens[s]) - 1
        blk = int(c.block_table[s, P // 16])
        expect[blk, P % 16] = kn[s]
    assert torch.equal(dc.K[0], expect)


def test_bad_block_id_is_reported_not_dereferenced(zp):
    c = zp_inputs.make_paged_case(12, 3, 32, 8, 128, 16, lens=[40, 20, 33], dtype="bf16")
    dc = DeviceCase(c)
    dc.table[1, 0] = c.n_total + 5  # out of range: must be skipped and flagged
    zp.zp_device_status(clear=True)
    out = torch.empty_like(dc.q)
    zp.zp_paged_decode_attn(_desc(zp, c), dc.q, dc.K[0], dc.V[0], dc.table, dc.lens, out)
    torch.cuda.synchronize()
    code, detail = zp.zp_device_status(clear=True)
    assert code == 7
    got = out.float().cpu().numpy()
    _check_out(got, c, dc.np_k(), dc.np_v(), [0, 2])  # other sequences unaffected


def test_workspace_too_small_is_rejected(zp):
    c = zp_inputs.make_paged_case(13, 2, 32, 8, 128, 16, lens=[40, 20], dtype="bf16")
    dc = DeviceCase(c)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(zp.ZPError) as e:
        zp.zp_paged_decode_attn(_desc(zp, c), dc.q, dc.K[0], dc.V[0], dc.table, dc.lens,
                                torch.empty_like(dc.q), workspace=ws)
    assert e.value.status == 4


def test_wait_that_runs_out_is_reported(zp):
    """Failure detection without a fault: the per-sequence control word of the
    in-kernel merge (the first 8 bytes per sequence of the decode workspace)
    is preset to a tagged arrival count that the CTAs' arrivals can never
    complete, so nobody publishes the cut sequence and every CTA that waits
    for it gives up after its 1 s limit.  The call returns, the device status
    reads ZP_ERR_TIMEOUT, and a cleared workspace decodes correctly again."""
    c = zp_inputs.make_paged_case(14, 1, 32, 8, 128, 16, lens=[8190], dtype="bf16")  # cut across all CTAs
    dc = DeviceCase(c)
    desc = _desc(zp, c)
    ws = torch.zeros(zp.zp_decode_workspace_size(desc, 1, dc.table.shape[1]), dtype=torch.uint8, device="cuda")
    tag = 0xC0DE5EC7A11D
    word = (tag << 16) | 0x4000  # phase 0, 16384 arrivals already counted
    ws[:8].view(torch.int64)[0] = word - (1 << 64) if word >= 1 << 63 else word  # same 64 bits
    S = torch.zeros(1, 8, dc.table.shape[1] * 16, device="cuda")
    zp.zp_device_status(clear=True)
    out = torch.empty_like(dc.q)
    zp.zp_paged_decode_attn(desc, dc.q, dc.K[0], dc.V[0], dc.table, dc.lens, out, score_accum=S, window=16,
                            workspace=ws)
    torch.cuda.synchronize()
    code, detail = zp.zp_device_status(clear=True)
    assert code == 6 and detail == 50
    ws.zero_()
    out = torch.empty_like(dc.q)
    zp.zp_paged_decode_attn(desc, dc.q, dc.K[0], dc.V[0], dc.table, dc.lens, out, score_accum=S, window=16,
                            workspace=ws)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    _check_out(out.float().cpu().numpy(), c, dc.np_k(), dc.np_v(), [0])


def _stale_scores(c, b, seed):
    """A stale score row per sequence (device) and the oracle's paged copy."""
    B, h_kv = c.seq_lens.shape[0], c.h_kv
    stride = c.block_table.shape[1]
    S0 = torch.rand(B, h_kv, stride * b, generator=torch.Generator().manual_seed(seed)) + 0.5
    S_ref = np.zeros((c.n_total, b, h_kv))
    for s in range(B):
        L = int(c.seq_lens[s])
        t = np.arange(L)
        S_ref[c.block_table[s].numpy()[t // b], t % b] = S0[s, :, :L].numpy().astype(np.float64).T
    return S0.cuda(), S_ref


@pytest.mark.parametrize("h_q,h_kv,d", [(32, 8, 128), (16, 4, 128), (8, 2, 64), (4, 1, 64)])
def test_window_score_step_with_two_cut_sequences_per_cta(zp, h_q, h_kv, d):
    """One decode step with the window score on the tensor-core path, with
    enough sequences that most CTAs hold the end of one sequence and the start
    of the next (two cut sequences per CTA: their merges and scores run side by
    side for h_kv >= 4, one after the other below) and one long sequence cut
    across about fifteen CTAs.  S starts stale: each token's piece is added to
    it, or written where the step is the first window row (App. C.2)."""
    b, w = 16, 16
    rng = np.random.default_rng(1234 + h_kv)
    lens = [int(x) for x in rng.integers(60, 400, size=119)] + [3001]
    lens[0], lens[7], lens[50] = 17, 161, 33  # L = 16 j + 1: the first window row (written)
    c = zp_inputs.make_paged_case(90 + h_kv, len(lens), h_q, h_kv, d, b, lens=lens, dtype="bf16")
    dc = DeviceCase(c)
    S, S_ref = _stale_scores(c, b, 11 + h_kv)
    got = _run_decode(zp, dc, score=S, window=w)
    K, V = dc.np_k(), dc.np_v()
    ref, probs = oracle.decode_attention(c.q.float().numpy(), K, V, c.block_table.numpy(), c.seq_lens.numpy(),
                                         want_probs=True)
    np.testing.assert_allclose(got, ref, **TOL_OUT["bf16"])
    oracle.accumulate_window_score(probs, c.block_table.numpy(), c.seq_lens.numpy(), h_kv, b, w, S_ref)
    Sg = S.cpu().numpy().astype(np.float64)
    for s, L in enumerate(lens):
        np.testing.assert_allclose(Sg[s, :, :L], gather_slots(S_ref, c.block_table[s].numpy(), L, b),
                                   **TOL_SCORE["bf16"])


def test_window_score_step_segments_beyond_the_prefetch_area(zp):
    """A layer of ~9k-token sequences (about 1,400 scored tokens per CTA): a
    CTA's logits rows no longer fit the stage area at once, so the window score
    takes them in chunks (score_segment); outputs of every sequence, scores of
    sampled ones against the oracle, S stale as above."""
    b, w = 16, 16
    c = zp_inputs.make_paged_case(1077, 24, 32, 8, 128, b, len_range=(8000, 10000), dtype="bf16")
    dc = DeviceCase(c)
    S, S_ref = _stale_scores(c, b, 17)
    got = _run_decode(zp, dc, score=S, window=w)
    seqs = [0, 5, 11, 16, 23]
    K, V = dc.np_k(), dc.np_v()
    _check_out(got, c, K, V, seqs)
    _, probs = oracle.decode_attention(c.q.float().numpy()[seqs], K, V, c.block_table.numpy()[seqs],
                                       c.seq_lens.numpy()[seqs], want_probs=True)
    oracle.accumulate_window_score(probs, c.block_table.numpy()[seqs], c.seq_lens.numpy()[seqs], 8, b, w, S_ref)
    Sg = S.cpu().numpy().astype(np.float64)
    for s in seqs:
        L = int(c.seq_lens[s])
        np.testing.assert_allclose(Sg[s, :, :L], gather_slots(S_ref, c.block_table[s].numpy(), L, b),
                                   **TOL_SCORE["bf16"])
