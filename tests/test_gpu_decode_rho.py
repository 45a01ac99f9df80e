"""GPU parity of the lightning redundancy computed inside the decode
[Zipage App. C.5 definition, C.7 same-block pairs] and of the compression
that takes it (zp_paged_decode_attn_rho, zp_compress_layers_rho).

* The decode's outputs and window scores stay those of the plain decode when
  it also forms the row sums (up to rounding: its stream-K split weighs the
  units that form them more, which moves the points where sequences are cut
  between CTAs and so the order of the partial merges); the row sums equal,
  bit for bit, those the compression's own kernel (zp_score_tokens) forms
  from the same keys, and the oracle's within the fp32 tolerance --
  including partial last blocks and a negative threshold, where rows past
  the block's end must take no part in the newest-row rule.
* After the same decode, compress_rho equals compress: keep sets, final
  scores, every K/V byte, F and the score rows bit-exact, first and later
  compressions, in-place and fresh targets, one and two layers per call.
"""
import numpy as np
import pytest
import torch

import oracle
import zp_inputs
from tests.gpu_util import DeviceCase

pytestmark = pytest.mark.gpu

RHO_TOL = dict(rtol=1e-4, atol=1e-4)  # fp32 sums of at most 16 cosines


@pytest.fixture(scope="module")
def zp():
    import compressed_paged_kv_zp_gb300 as m
    return m


def _desc(zp, c):
    return zp.cache_desc(c.h_q, c.h_kv, c.d, c.b, c.n_total, torch.bfloat16 if c.dtype == "bf16" else torch.float32)


def _keys(K0, table_row, L, h, b=16):
    t = np.arange(L)
    return np.ascontiguousarray(K0[np.asarray(table_row)[t // b], t % b, h], dtype=np.float32)


def _score_tokens_rho(zp, desc, K, table, lens, p):
    """rho of zp_score_tokens (lightning) for these sequences, from its workspace."""
    n, h_kv = int(table.shape[0]), desc.h_kv
    Lmax = int(lens.max().item())
    S = torch.full((n, h_kv, Lmax), 0.01, device="cuda")
    F = torch.zeros(desc.n_total_blocks, desc.block_size, h_kv, device="cuda")
    first = torch.ones(n, dtype=torch.uint8, device="cuda")
    scores = torch.empty((n, h_kv, Lmax), device="cuda")
    ws = torch.empty(zp.zp_score_workspace_size(desc, n, Lmax), dtype=torch.uint8, device="cuda")
    params = zp.score_params(window=1, lightning=True, threshold=p)
    zp.zp_score_tokens(desc, params, K, table, lens, first, S, F, scores, workspace=ws)
    torch.cuda.synchronize()
    assert zp.zp_device_status() == (0, 0)
    off = (n * h_kv * Lmax * 4 + 255) // 256 * 256
    return ws[off:off + n * h_kv * Lmax * 4].view(torch.float32).view(n, h_kv, Lmax).cpu().numpy()


@pytest.mark.parametrize("p", [0.5, -0.3])
def test_decode_rho_equals_compression_rho_and_oracle(zp, p):
    B, h_q, h_kv, d, b, w = 10, 32, 8, 128, 16, 16
    lens = [1, 16, 17, 33, 250, 511, 512, 1000, 1407, 2049]
    c = zp_inputs.make_paged_case(4100, B, h_q, h_kv, d, b, lens=lens, dtype="bf16")
    zp_inputs.plant_duplicates(c, 4101)
    desc = _desc(zp, c)
    table_stride = int(c.block_table.shape[1])
    slot = np.full(B, -1, np.int32)
    chosen = [0, 2, 3, 5, 6, 8, 9]
    for j, s in enumerate(chosen):
        slot[s] = len(chosen) - 1 - j  # permuted rows
    rows = torch.from_numpy(slot).cuda()
    stride = max(lens) + 5
    res = {}
    for mode in ("plain", "rho"):
        dc = DeviceCase(c)
        out = torch.empty(B, h_q, d, dtype=torch.bfloat16, device="cuda")
        S = torch.full((B, h_kv, table_stride * b), 0.125, device="cuda")
        rho = torch.full((len(chosen), h_kv, stride), -9.0, device="cuda")
        if mode == "plain":
            zp.zp_paged_decode_attn(desc, dc.q, dc.K[0], dc.V[0], dc.table, dc.lens, out, S, w)
        else:
            zp.zp_paged_decode_attn(desc, dc.q, dc.K[0], dc.V[0], dc.table, dc.lens, out, S, w, rho=rho,
                                    rho_rows=rows, rho_threshold=p)
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        res[mode] = (out.cpu(), S.cpu(), rho.cpu().numpy())
    # outputs (bf16: one unit in the last place) and window scores (fp32 sums)
    torch.testing.assert_close(res["rho"][0].float(), res["plain"][0].float(), atol=1e-2, rtol=1e-2)
    torch.testing.assert_close(res["rho"][1], res["plain"][1], atol=1e-9, rtol=1e-5)
    rho = res["rho"][2]
    # the compression's own kernel on the same keys
    sub = torch.tensor(chosen, dtype=torch.long)
    dc = DeviceCase(c)
    ref_gpu = _score_tokens_rho(zp, desc, dc.K[0], dc.table[sub.cuda()].contiguous(), dc.lens[sub.cuda()].contiguous(),
                                p)
    K0 = c.k_cache[0].float().numpy()
    for j, s in enumerate(chosen):
        L = lens[s]
        r = slot[s]
        assert np.array_equal(rho[r, :, :L], ref_gpu[j, :, :L]), s
        assert (rho[r, :, L:] == -9.0).all()  # nothing past L
        for h in range(h_kv):
            want = oracle.redundancy_rho(_keys(K0, c.block_table[s].numpy(), L, h), b, p, True)
            np.testing.assert_allclose(rho[r, h, :L], want, **RHO_TOL)


@pytest.mark.parametrize("dtype,p", [("bf16", -0.3), ("f32", -0.3), ("f32", 0.5)])
def test_lightning_partial_last_block_matches_oracle(zp, dtype, p):
    """zp_score_tokens' lightning row sums on lengths that end inside a block
    (nvalid < b), also with p < 0 where the zero entries of the missing rows
    would exceed the threshold."""
    B, h_q, h_kv, d, b = 5, 8, 2, 64, 16
    lens = [3, 17, 40, 95, 130]
    c = zp_inputs.make_paged_case(4200, B, h_q, h_kv, d, b, lens=lens, dtype=dtype)
    zp_inputs.plant_duplicates(c, 4201)
    desc = _desc(zp, c)
    dc = DeviceCase(c)
    rho = _score_tokens_rho(zp, desc, dc.K[0], dc.table, dc.lens, p)
    K0 = c.k_cache[0].float().numpy()
    for s, L in enumerate(lens):
        for h in range(h_kv):
            want = oracle.redundancy_rho(_keys(K0, c.block_table[s].numpy(), L, h), b, p, True)
            np.testing.assert_allclose(rho[s, h, :L], want, **RHO_TOL)


@pytest.mark.parametrize("layers", [1, 2])
def test_compress_with_decode_rho_equals_compress(zp, layers):
    """decode_rho -> compress against decode_rho -> compress_rho, each pair
    back to back on one stream (the compression launched as a programmatic
    dependent of the decode), on copies of the same state."""
    B, h_q, h_kv, d, b, w, N_max = 9, 32, 8, 128, 16, 16, 8
    g = torch.Generator().manual_seed(4300 + layers)
    lens = ((torch.randint(200, 1200, (B,), generator=g) // b) * b).tolist()
    c = zp_inputs.make_paged_case(4300 + layers, B, h_q, h_kv, d, b, lens=lens, dtype="bf16", layers=layers,
                                  spare_blocks=B * N_max)
    zp_inputs.plant_duplicates(c, 4310)
    desc = _desc(zp, c)
    table_stride = int(c.block_table.shape[1])
    chosen = [1, 2, 4, 7, 8]
    n = len(chosen)
    k = (N_max - 1) * b
    Lmax = max(lens[s] for s in chosen)
    rng = np.random.default_rng(4320 + layers)
    S0 = (rng.random((layers, B, h_kv, table_stride * b)) / 100).astype(np.float32)
    F0 = (rng.random((layers, c.n_total, b, h_kv)) / 80).astype(np.float32)
    first = torch.tensor([1, 0, 0, 1, 0], dtype=torch.uint8, device="cuda")
    free = c.free_blocks.numpy()
    tg = np.stack([free[i * (N_max - 1):(i + 1) * (N_max - 1)] if i % 2 else c.block_table[s, : N_max - 1].numpy()
                   for i, s in enumerate(chosen)]).astype(np.int32)
    targets = torch.from_numpy(tg).cuda()
    sub = torch.tensor(chosen, dtype=torch.long, device="cuda")
    slot = np.full(B, -1, np.int32)
    slot[chosen] = np.arange(n, dtype=np.int32)
    dec_rows = torch.from_numpy(slot).cuda()
    attn_rows = torch.tensor(chosen, dtype=torch.int32, device="cuda")
    params = zp.score_params(window=w, threshold=0.5)
    res = {}
    for mode in ("plain", "rho"):
        dc = DeviceCase(c)
        S = torch.from_numpy(S0.copy()).cuda()
        F = torch.from_numpy(F0.copy()).cuda()
        out = torch.empty(layers, B, h_q, d, dtype=torch.bfloat16, device="cuda")
        rho = torch.full((layers, n, h_kv, Lmax), -9.0, device="cuda")
        keep = torch.empty(layers, n, h_kv, k, dtype=torch.int32, device="cuda")
        scores = torch.full((layers, n, h_kv, Lmax), -5.0, device="cuda")
        tab, ln = dc.table[sub].contiguous(), dc.lens[sub].contiguous()
        for l in range(layers):
            zp.zp_paged_decode_attn(desc, dc.q, dc.K[l], dc.V[l], dc.table, dc.lens, out[l], S[l], w,
                                    rho=rho[l], rho_rows=dec_rows, rho_threshold=0.5)
        Kx, Vx, Sx, Fx = (dc.K, dc.V, S, F) if layers > 1 else (dc.K[0], dc.V[0], S[0], F[0])
        kx, sx = (keep, scores) if layers > 1 else (keep[0], scores[0])
        if mode == "plain":
            zp.zp_compress_layers(desc, params, Kx, Vx, tab, ln, first, Sx, Fx, targets, k, kx, Lmax, rows=attn_rows,
                                  scores_out=sx)
        else:
            zp.zp_compress_layers(desc, params, Kx, Vx, tab, ln, first, Sx, Fx, targets, k, kx, Lmax, rows=attn_rows,
                                  scores_out=sx, rho=rho if layers > 1 else rho[0])
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        res[mode] = [t.cpu() for t in (out, S, F, keep, scores, dc.K, dc.V)]
    names = ("out", "S", "F", "keep", "scores", "K", "V")
    for nm, x, y in zip(names, res["plain"], res["rho"]):
        assert torch.equal(x, y), nm
    # the compression did act: the moved rows of the fresh targets are the kept tokens' rows
    K0 = c.k_cache[0].float().numpy()
    Kf = res["rho"][5][0].float().numpy()
    kp = res["rho"][3][0].numpy()
    for i, s in enumerate(chosen):
        if i % 2:
            for h in range(h_kv):
                for r in range(0, k, 13):
                    pos = kp[i, h, r]
                    assert np.array_equal(Kf[tg[i, r // b], r % b, h], K0[c.block_table[s, pos // b], pos % b, h])


def test_rho_paths_refuse_what_they_do_not_cover(zp):
    B, h_q, h_kv, d, b = 2, 8, 2, 64, 16
    c = zp_inputs.make_paged_case(4400, B, h_q, h_kv, d, b, lens=[32, 48], dtype="f32")
    desc = _desc(zp, c)
    dc = DeviceCase(c)
    out = torch.empty(B, h_q, d, device="cuda")
    rho = torch.zeros(B, h_kv, 64, device="cuda")
    rows = torch.arange(B, dtype=torch.int32, device="cuda")
    with pytest.raises(zp.ZPError) as e:  # fp32 cache: no tensor-core decode
        zp.zp_paged_decode_attn(desc, dc.q, dc.K[0], dc.V[0], dc.table, dc.lens, out, rho=rho, rho_rows=rows)
    assert e.value.status == 2
    cb = zp_inputs.make_paged_case(4401, B, 32, 8, 128, b, lens=[32, 48], dtype="bf16", spare_blocks=8)
    descb = _desc(zp, cb)
    dcb = DeviceCase(cb)
    S = torch.zeros(B, 8, 64, device="cuda")
    F = torch.zeros(cb.n_total, b, 8, device="cuda")
    keep = torch.empty(B, 8, 16, dtype=torch.int32, device="cuda")
    first = torch.ones(B, dtype=torch.uint8, device="cuda")
    tg = cb.block_table[:, :1].contiguous().cuda()
    with pytest.raises(zp.ZPError) as e:  # all-pairs redundancy: the row sums are not lightning's
        zp.zp_compress_layers(descb, zp.score_params(window=16, lightning=False), dcb.K[0], dcb.V[0], dcb.table,
                              dcb.lens, first, S, F, tg, 16, keep, 48, rho=torch.zeros(B, 8, 64, device="cuda"))
    assert e.value.status == 2


@pytest.mark.parametrize("B,h_q,h_kv,d,lo,hi,every", [
    (300, 32, 8, 128, 17, 300, 1),   # every sequence forms row sums: several 32-wide scan rounds
    (2500, 4, 1, 64, 3, 40, 3),      # the split's arrays do not fit the stage area: unweighted split
])
def test_decode_rho_many_sequences(zp, B, h_q, h_kv, d, lo, hi, every):
    """Row sums for many sequences at once: the decode's outputs stay those of
    the plain decode (rounding) and every row equals the compression's own
    kernel; sampled rows against the oracle."""
    b, w = 16, 16
    g = torch.Generator().manual_seed(4500 + B)
    lens = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    c = zp_inputs.make_paged_case(4500 + B, B, h_q, h_kv, d, b, lens=lens, dtype="bf16")
    zp_inputs.plant_duplicates(c, 4501)
    desc = _desc(zp, c)
    table_stride = int(c.block_table.shape[1])
    chosen = list(range(0, B, every))
    slot = np.full(B, -1, np.int32)
    slot[chosen] = np.arange(len(chosen), dtype=np.int32)
    rows = torch.from_numpy(slot).cuda()
    stride = max(lens)
    res = {}
    for mode in ("plain", "rho"):
        dc = DeviceCase(c)
        out = torch.empty(B, h_q, d, dtype=torch.bfloat16, device="cuda")
        S = torch.zeros(B, h_kv, table_stride * b, device="cuda")
        rho = torch.full((len(chosen), h_kv, stride), -9.0, device="cuda")
        extra = dict(rho=rho, rho_rows=rows, rho_threshold=0.5) if mode == "rho" else {}
        zp.zp_paged_decode_attn(desc, dc.q, dc.K[0], dc.V[0], dc.table, dc.lens, out, S, w, **extra)
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        res[mode] = (out.cpu(), S.cpu(), rho.cpu().numpy())
    torch.testing.assert_close(res["rho"][0].float(), res["plain"][0].float(), atol=1e-2, rtol=1e-2)
    torch.testing.assert_close(res["rho"][1], res["plain"][1], atol=1e-9, rtol=1e-5)
    rho = res["rho"][2]
    sub = torch.tensor(chosen, dtype=torch.long, device="cuda")
    dc = DeviceCase(c)
    ref_gpu = _score_tokens_rho(zp, desc, dc.K[0], dc.table[sub].contiguous(), dc.lens[sub].contiguous(), 0.5)
    K0 = c.k_cache[0].float().numpy()
    for j, s in enumerate(chosen):
        L = lens[s]
        assert np.array_equal(rho[j, :, :L], ref_gpu[j, :, :L]), s
    for j in range(0, len(chosen), max(1, len(chosen) // 12)):
        s, L = chosen[j], lens[chosen[j]]
        for h in range(h_kv):
            want = oracle.redundancy_rho(_keys(K0, c.block_table[s].numpy(), L, h), b, 0.5, True)
            np.testing.assert_allclose(rho[j, h, :L], want, **RHO_TOL)
