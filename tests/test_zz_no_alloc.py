"""mla_decode_latent_noalloc: the decode entry point for callers that cannot allocate.

Some callers are handed only their input and output buffers (for example a plugin inside
a host runtime that offers no device allocator) or must not call cudaMalloc in their
loop.  For them the library keeps the split-KV partials in a fixed array of
MLA_NOALLOC_SCRATCH_BYTES instead of a workspace.  These tests call that entry point
through the C ABI and check that it gives what mla_decode_latent (with a workspace)
gives, bit for bit, on two calls in a row with different shapes, so that whatever the
first call left in the shared array cannot leak into the second.  This file sorts last so that a
run stopping at the first failure has run every other test before it.
"""
import ctypes

import pytest
import torch

from mla_latent_kv_70_b300 import inputs as I
from tests.mla_cases import DeviceCase

LIMIT = 32 << 20        # MLA_NOALLOC_SCRATCH_BYTES in include/mla.h
P = 4096                # a fake aligned address: a rejected call never dereferences it


@pytest.fixture(scope="module")
def lib():
    import mla_latent_kv_70_b300 as mla
    from mla_latent_kv_70_b300 import build
    build.build()
    return mla.lib()


def noalloc_args(**over):
    a = dict(q_cat=P, kv=P, kv_seq_stride=4096, seqlens=P, block_table=None, max_pages=0,
             page_size=64, num_pages=0, B=64, S=1, H=128, causal=0, scale=0.07, num_splits=1,
             max_seqlen=4096, o_lat=P, lse=P, status=None, stream=None)
    a.update(over)
    return list(a.values())


def test_noalloc_rejects_on_the_host(lib):
    # Every check of mla_decode_latent runs before the scratch address is looked up, so
    # none of these calls makes a CUDA call (the fake pointers are never dereferenced).
    assert lib.mla_decode_latent_noalloc(*noalloc_args(q_cat=None)) == 1
    assert lib.mla_decode_latent_noalloc(*noalloc_args(num_splits=200)) == 1
    assert lib.mla_decode_latent_noalloc(*noalloc_args(q_cat=P + 2)) == 1      # misaligned
    assert lib.mla_decode_latent_noalloc(*noalloc_args(H=8)) == 2              # unsupported
    assert lib.mla_decode_latent_noalloc(*noalloc_args(scale=0.0)) == 1
    assert lib.mla_decode_latent_noalloc(*noalloc_args(kv_seq_stride=100)) == 1
    # 128 splits of 64 x 128 rows need 2.15 GB of partials: beyond the fixed array.
    assert lib.mla_decode_workspace_bytes(64, 1, 128, 128, 4096) > LIMIT
    assert lib.mla_decode_latent_noalloc(*noalloc_args(num_splits=128)) == 4


def ptr(t):
    return None if t is None else t.data_ptr()


@pytest.mark.gpu
def test_noalloc_matches_decode_latent_twice(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_latent_kv_70_b300 as mla
    calls = [
        (I.make_case("noalloc_contig", 2, 1, 128, [3000, 4096], seed=21), 8),
        (I.make_case("noalloc_paged", 3, 2, 128, [700, 64, 1500], paged=True, causal=True,
                     seed=22), 5),
    ]
    for case, splits in calls:
        dc = DeviceCase(case)
        B, S, H = case.B, case.S, case.H
        max_seqlen = max(case.seqlens)
        need = mla.mla_decode_workspace_bytes(B, S, H, splits, max_seqlen)
        assert 0 < need <= LIMIT
        q_cat = torch.empty(B, S, H, 576, dtype=torch.bfloat16, device="cuda")
        mla.mla_absorb_q(dc.q_nope, dc.q_rope, dc.w_uk, None, case.theta, q_cat)
        # The existing entry point, with a workspace the test allocates.
        ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
        ref_o = torch.empty(B, S, H, 512, device="cuda")
        ref_l = torch.empty(B, S, H, device="cuda")
        mla.mla_decode_latent(q_cat, dc.kv, dc.seqlens, ref_o, ref_l, scale=case.scale,
                              max_seqlen=max_seqlen, block_table=dc.block_table,
                              causal=case.causal, num_splits=splits, workspace=ws)
        # The allocation-free entry point, called directly through the C ABI.
        o = torch.full((B, S, H, 512), float("nan"), device="cuda")
        lse = torch.full((B, S, H), float("nan"), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        bt = dc.block_table
        stride = 0 if case.paged else dc.kv.shape[1]
        rc = lib.mla_decode_latent_noalloc(
            ptr(q_cat), ptr(dc.kv), stride, ptr(dc.seqlens), ptr(bt),
            0 if bt is None else bt.shape[1], 64, dc.kv.shape[0] if case.paged else 0,
            B, S, H, int(case.causal), ctypes.c_float(case.scale), splits, max_seqlen,
            ptr(o), ptr(lse), ptr(status), torch.cuda.current_stream().cuda_stream)
        assert rc == 0, mla.mla_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.isfinite(o).all()
        # The same kernels with the same split plan: bit for bit the same results.
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l), case.name
