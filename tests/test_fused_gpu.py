"""GPU parity of the pre-fused weights ([CALC] "Query·출력 투영과 합치기") through the C ABI:
the offline products W_UQ W_UK^T and W_UV W_O, the key absorption from the query latent,
the output projection summed over heads, and a whole decode step on the fused weights
against the oracle's unfused definition."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from mla_latent_kv_70_b300 import inputs as I
from tests.mla_cases import ROW_REL_TOL, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_70_b300 import build
    build.build()


def fp32_sum_bound(a_abs, b_abs, n):
    """fp32 accumulation of n products: at most n * 2^-24 of the sum of their magnitudes."""
    return n * 2.0 ** -24 * (a_abs @ b_abs)


@pytest.mark.parametrize("H,d_cq,d_model", [(16, 1536, 4096), (32, 192, 256)])
def test_fuse_weights_match_oracle(H, d_cq, d_model):
    import mla_latent_kv_70_b300 as mla
    case = I.make_case("fuse", 1, 1, H, [1], seed=81)
    w_uk, w_uv = I.weights(case)
    w_uq, w_o = I.query_side_weights(case, d_cq), I.output_weights(case, d_model)
    w_uqk = torch.empty(H, d_cq, 512, dtype=torch.bfloat16, device="cuda")
    w_uvo = torch.empty(H, 512, d_model, dtype=torch.bfloat16, device="cuda")
    mla.mla_fuse_weights(w_uq.cuda(), w_uk.cuda(), w_uv.cuda(), w_o.cuda(), w_uqk, w_uvo)
    torch.cuda.synchronize()
    d = lambda t: t.double().numpy()
    ref_q = O.fuse_query_weights(d(w_uq), d(w_uk))
    ref_o = O.fuse_output_weights(d(w_uv), d(w_o))
    # bf16 output of an fp32 sum of 128 products: one bf16 rounding (unit roundoff 2^-8)
    # plus the fp32 accumulation error.
    for got, ref, acc in ((w_uqk, ref_q, np.einsum("hik,hck->hic", np.abs(d(w_uq)), np.abs(d(w_uk)))),
                          (w_uvo, ref_o, np.einsum("hcv,hvj->hcj", np.abs(d(w_uv)), np.abs(d(w_o))))):
        g = got.cpu().double().numpy()
        bound = 2.0 ** -8 * np.abs(ref) + 128 * 2.0 ** -24 * acc
        assert np.all(np.abs(g - ref) <= bound)


@pytest.mark.parametrize("B,S,H,rope", [(64, 1, 128, False), (5, 2, 16, True), (150, 2, 32, False)])
def test_absorb_q_fused_matches_oracle(B, S, H, rope):
    import mla_latent_kv_70_b300 as mla
    d_cq = I.D_CQ
    case = I.make_case("absorb_fused", B, S, H, [64] * B, seed=83)
    c_q = I.c_q(case, d_cq)
    # A seeded fused weight (this call is checked on its own): std sqrt(128 / (512 * d_cq)),
    # the spread of W_UQ W_UK^T for the weights above.
    w_uqk = I.randn_bf16((H, d_cq, 512), case.seed, "wuqk", 0, math.sqrt(128.0 / (512 * d_cq)))
    _, q_rope = I.queries(case)
    q_pos = case.q_positions() if rope else None
    q_cat = torch.empty(B, S, H, 576, dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_q_fused(c_q.cuda(), q_rope.cuda(), w_uqk.cuda(), None if q_pos is None else q_pos.cuda(),
                           1e4, q_cat)
    torch.cuda.synchronize()
    got = q_cat.cpu().double().numpy()
    cq, w = c_q.double().numpy(), w_uqk.double().numpy()
    ref = O.absorb_q_from_latent(cq, w)
    bound = 2.0 ** -8 * np.abs(ref) + d_cq * 2.0 ** -24 * O.absorb_q_from_latent(np.abs(cq), np.abs(w))
    assert np.all(np.abs(got[..., :512] - ref) <= bound)
    qr = q_rope.double().numpy()
    if rope:
        ref_r = O.rope_interleaved(qr, q_pos.double().numpy()[..., None], 1e4)
        np.testing.assert_allclose(got[..., 512:], ref_r, rtol=2 ** -7, atol=2 ** -7)
    else:
        np.testing.assert_array_equal(got[..., 512:], qr)


@pytest.mark.parametrize("B,S,H,d_model", [(64, 1, 128, 4096), (3, 2, 16, 256)])
def test_out_proj_fused_matches_oracle(B, S, H, d_model):
    import mla_latent_kv_70_b300 as mla
    case = I.make_case("out_fused", B, S, H, [64] * B, seed=85)
    o_lat = torch.randn(B, S, H, 512, generator=torch.Generator().manual_seed(4))
    w_uvo = I.randn_bf16((H, 512, d_model), case.seed, "wuvo", 0, 1.0 / math.sqrt(H * 512))
    out = torch.empty(B, S, d_model, device="cuda")
    ws = torch.empty(mla.mla_out_proj_fused_workspace_bytes(B, S, H), dtype=torch.uint8, device="cuda")
    mla.mla_out_proj_fused(o_lat.cuda(), w_uvo.cuda(), out, ws)
    torch.cuda.synchronize()
    lat, w = o_lat.double().numpy(), w_uvo.double().numpy()
    ref = O.out_proj_fused(lat, w)
    got = out.cpu().numpy()
    assert row_rel_err(got, ref) <= ROW_REL_TOL
    # o_lat is rounded to bf16 on its way to the tensor core (2^-8 of each product), and
    # the H*512 products are summed in fp32 in parts: twice the first, plus the second.
    mag = O.out_proj_fused(np.abs(lat), np.abs(w))
    bound = 2.0 ** -7 * mag + H * 512 * 2.0 ** -24 * mag
    assert np.all(np.abs(got - ref) <= bound + 1e-6)


def test_decode_step_on_fused_weights_matches_unfused_oracle():
    # c^Q -> (W_UQ W_UK^T) -> latent attention -> (W_UV W_O), every product on the GPU,
    # against the oracle's unfused definition: q_nope = c^Q W_UQ, expanded attention per
    # head, out = sum_h o_h W_O[h].
    import mla_latent_kv_70_b300 as mla
    lens = [300, 77, 1000, 5]
    case = I.make_case("fused_step", len(lens), 1, 16, lens, seed=87)
    d_cq, d_model = I.D_CQ, 1024
    kv = I.cache(case, device="cuda")
    w_uk, w_uv = I.weights(case)
    w_uq, w_o = I.query_side_weights(case, d_cq), I.output_weights(case, d_model)
    c_q = I.c_q(case, d_cq)
    _, q_rope = I.queries(case)
    H, B = case.H, case.B
    w_uqk = torch.empty(H, d_cq, 512, dtype=torch.bfloat16, device="cuda")
    w_uvo = torch.empty(H, 512, d_model, dtype=torch.bfloat16, device="cuda")
    mla.mla_fuse_weights(w_uq.cuda(), w_uk.cuda(), w_uv.cuda(), w_o.cuda(), w_uqk, w_uvo)
    q_cat = torch.empty(B, 1, H, 576, dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_q_fused(c_q.cuda(), q_rope.cuda(), w_uqk, None, 1e4, q_cat)
    o_lat = torch.empty(B, 1, H, 512, device="cuda")
    lse = torch.empty(B, 1, H, device="cuda")
    seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    mla.mla_decode_latent(q_cat, kv, seqlens, o_lat, lse, scale=case.scale, max_seqlen=max(lens), num_splits=1)
    out = torch.empty(B, 1, d_model, device="cuda")
    ws = torch.empty(mla.mla_out_proj_fused_workspace_bytes(B, 1, H), dtype=torch.uint8, device="cuda")
    mla.mla_out_proj_fused(o_lat, w_uvo, out, ws)
    torch.cuda.synchronize()
    d = lambda t: t.double().numpy()
    wq, wk, wv, wo = d(w_uq), d(w_uk), d(w_uv), d(w_o)
    for b, T in enumerate(lens):
        rows = I.seq_rows(case, b)[:T].double().numpy()
        q_nope = np.einsum("si,hik->shk", d(I.seq_c_q(case, b, d_cq)), wq)
        o, _ = O.decode_expanded_seq(q_nope, d(I.seq_queries(case, b)[1]), rows[:, :512], rows[:, 512:],
                                     wk, wv, case.scale)
        ref = O.out_proj_heads(o, wo)
        assert row_rel_err(out[b].cpu().numpy(), ref) <= ROW_REL_TOL, b
