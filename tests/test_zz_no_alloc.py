"""The decode entry point that allocates nothing (zp_paged_decode_attn_noalloc).

Some callers cannot hand the library a workspace: a serving loop whose device
memory is all reserved up front may not call cudaMalloc between steps, and a
plain C client of the library may have no device allocator at all.  For
them the library keeps one fixed scratch array on each GPU.  This test calls
that entry point through the C ABI twice in a row on the same inputs and
checks both results (attention output and window score) against the ordinary
entry point with a caller workspace, at the tolerances of the other decode
tests.  The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import zp_inputs
from tests.gpu_util import TOL_OUT, TOL_SCORE

pytestmark = pytest.mark.gpu


def _args(zp, c, dev):
    desc = zp.cache_desc(c.h_q, c.h_kv, c.d, c.b, c.n_total, torch.bfloat16)
    K = c.k_cache[0].contiguous().to(dev)
    V = c.v_cache[0].contiguous().to(dev)
    return desc, c.q.to(dev), K, V, c.block_table.to(dev), c.seq_lens.to(dev)


def test_noalloc_decode_matches_workspace_decode_twice():
    import compressed_paged_kv_zp_gb300 as zp
    dev = torch.device("cuda")
    c = zp_inputs.make_paged_case(2024, 24, 32, 8, 128, 16, len_range=(1, 1500), dtype="bf16")
    desc, q, K, V, table, lens = _args(zp, c, dev)
    S_ref = torch.zeros(c.B, 8, table.shape[1] * 16, device=dev)
    out_ref = torch.empty_like(q)
    zp.zp_paged_decode_attn(desc, q, K, V, table, lens, out_ref, score_accum=S_ref, window=16)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        S = torch.zeros(c.B, 8, table.shape[1] * 16, device=dev)
        rc = zp.lib.zp_paged_decode_attn_noalloc(
            ctypes.byref(desc), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(K.data_ptr()),
            ctypes.c_void_p(V.data_ptr()), ctypes.c_void_p(table.data_ptr()), table.shape[1],
            ctypes.c_void_p(lens.data_ptr()), c.B, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(S.data_ptr()), None, 0, 16, stream)
        assert rc == 0, zp.lib.zp_last_error().decode()
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        torch.testing.assert_close(out.float(), out_ref.float(), **TOL_OUT["bf16"])
        torch.testing.assert_close(S, S_ref, **TOL_SCORE["bf16"])


def test_noalloc_starts_clean_after_a_stale_control_word():
    """A call that gave up on its bounded wait can leave a control word of the
    built-in array counting arrivals that never completed, and a caller of this
    entry point cannot reach the array to clear it.  The test writes such a word
    (phase 0, 16384 arrivals) for a sequence cut across every CTA; the next call
    must clear it itself: no ZP_ERR_TIMEOUT, the same result as the workspace
    decode, and again on the call after."""
    import compressed_paged_kv_zp_gb300 as zp
    dev = torch.device("cuda")
    c = zp_inputs.make_paged_case(14, 1, 32, 8, 128, 16, lens=[8190], dtype="bf16")
    desc, q, K, V, table, lens = _args(zp, c, dev)
    out_ref = torch.empty_like(q)
    zp.zp_paged_decode_attn(desc, q, K, V, table, lens, out_ref)
    torch.cuda.synchronize()
    stale = (0xC0DE5EC7A11D << 16) | 0x4000
    zp.zp_device_status(clear=True)
    for call in range(2):
        rc = zp.lib.zp_debug_noalloc_preset_ctl(0, stale)
        assert rc == 0, zp.lib.zp_last_error().decode()
        out = torch.full_like(q, float("nan"))
        zp.zp_paged_decode_attn_noalloc(desc, q, K, V, table, lens, out)
        torch.cuda.synchronize()
        assert zp.zp_device_status() == (0, 0)
        torch.testing.assert_close(out.float(), out_ref.float(), **TOL_OUT["bf16"])


def test_noalloc_rejects_a_call_larger_than_its_buffer():
    import compressed_paged_kv_zp_gb300 as zp
    desc = zp.cache_desc(32, 8, 128, 16, 1000, torch.bfloat16)
    need = zp.zp_decode_workspace_size(desc, 4096, 4096)
    assert need > (64 << 20)
    q = torch.zeros(1, 32, 128, dtype=torch.bfloat16, device="cuda")
    table = torch.zeros(4096, 4096, dtype=torch.int32, device="cuda")
    lens = torch.ones(4096, dtype=torch.int32, device="cuda")
    with pytest.raises(zp.ZPError) as e:
        zp.zp_paged_decode_attn_noalloc(desc, q, q, q, table, lens, q)
    assert e.value.status == 4
