"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases are compared in full; the five named workloads run at their full sizes in
the launch configuration the bench uses, and are compared on seeded samples of
sequences (every head and every output of each sampled sequence).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from mla_latent_kv_70_b300 import inputs as I
from tests.mla_cases import (ROW_REL_TOL, DeviceCase, check_case, check_lse, lse_err,
                             lse_tolerance, oracle_seq, row_rel_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_70_b300 import build
    build.build()


# ----------------------------------------------------------------------------
# Small cases, compared in full
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("splits", [1, 2, 0])
def test_tiny_workload(splits):
    case = I.tiny()
    dc = DeviceCase(case)
    st = dc.step(num_splits=splits)
    check_case(dc, st, range(case.B), expanded_heads=list(range(case.H)))


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("splits", [1, 3, 64])
def test_ragged_contiguous_edges(H, splits):
    lens = [1, 5, 63, 64, 65, 200, 0, 129]
    case = I.make_case("edges", len(lens), 1, H, lens, t_cap=256, seed=3)
    dc = DeviceCase(case)
    for b, T in enumerate(lens):
        dc.kv[b, T:] = float("nan")       # rows past the sequence must never be used
    st = dc.step(num_splits=splits, max_seqlen=256)
    check_case(dc, st, range(case.B))
    assert np.all(st.o_lat[6].cpu().numpy() == 0)
    assert np.all(np.isneginf(st.lse[6].cpu().numpy()))


@pytest.mark.parametrize("splits", [1, 2])
def test_every_tile_count_up_to_13(splits):
    # The decode kernel cycles its barriers with period 6 tiles (three score groups, two
    # receive buffers, two rope and V slots, three score slots), and re-arms them by the
    # number of tiles left.  One sequence per tile count 1..13, with ragged last tiles and
    # NaN past the end, covers every residue twice.
    lens = [64 * n - (7 * n) % 64 for n in range(1, 14)]
    case = I.make_case("tile_counts", len(lens), 1, 128, lens, t_cap=13 * 64, seed=11)
    dc = DeviceCase(case)
    for b, T in enumerate(lens):
        dc.kv[b, T:] = float("nan")
    st = dc.step(num_splits=splits, max_seqlen=13 * 64)
    check_case(dc, st, range(case.B))


@pytest.mark.parametrize("splits", [1, 4])
def test_paged_small(splits):
    lens = [70, 1, 300, 64]
    case = I.make_case("paged_small", 4, 1, 128, lens, paged=True, seed=5)
    dc = DeviceCase(case)
    for b, T in enumerate(lens):
        last = int(case.block_table[b, case.pages_per_seq[b] - 1])
        off = T - (case.pages_per_seq[b] - 1) * 64
        dc.kv[last, off:] = float("nan")
    st = dc.step(num_splits=splits)
    check_case(dc, st, range(case.B))


def test_paged_equals_contiguous_bitwise():
    lens = [300, 77]
    paged = I.make_case("p", 2, 1, 128, lens, paged=True, seed=9)
    cont = I.make_case("c", 2, 1, 128, lens, seed=9, t_cap=320)
    dp, dcn = DeviceCase(paged), DeviceCase(cont)
    for b, T in enumerate(lens):
        rows = I.seq_rows(paged, b)[:T].cuda()
        dcn.kv[b, :T] = rows
    sp = dp.step(num_splits=2)
    sc = dcn.step(num_splits=2)
    assert torch.equal(sp.o_lat, sc.o_lat) and torch.equal(sp.lse, sc.lse)


@pytest.mark.parametrize("lens", [[100, 7, 2, 1], [129, 64]])
def test_causal_two_tokens_with_rope(lens):
    case = I.make_case("mtp_small", len(lens), 2, 128, lens, causal=True, rope=True, seed=11)
    dc = DeviceCase(case)
    st = dc.step(num_splits=1)
    check_case(dc, st, range(case.B), expanded_heads=[0, 77])
    st2 = dc.step(num_splits=3)
    check_case(dc, st2, range(case.B))


@pytest.mark.parametrize("S", [3, 4])
def test_causal_multi_token_with_rope(S):
    # The most query tokens per sequence the ABI accepts, end to end with RoPE.
    lens = [S, 40, 300]
    case = I.make_case("mtp_s%d" % S, len(lens), S, 128, lens, causal=True, rope=True, seed=51 + S)
    dc = DeviceCase(case)
    for splits in (1, 3):
        st = dc.step(num_splits=splits)
        check_case(dc, st, range(case.B), expanded_heads=[1, 100] if splits == 1 else None)


@pytest.mark.parametrize("splits", [1, 3])
def test_paged_causal_two_tokens_with_rope(splits):
    # Paged pool, causal pair of query tokens, k^R rotated through the block table.
    lens = [130, 2, 700, 64]
    case = I.make_case("paged_mtp", len(lens), 2, 128, lens, paged=True, causal=True, rope=True,
                       seed=57)
    dc = DeviceCase(case)
    st = dc.step(num_splits=splits)
    check_case(dc, st, range(case.B), expanded_heads=[9] if splits == 1 else None)


@pytest.mark.parametrize("H", [48, 112])
def test_mid_head_counts(H):
    # Head counts between the two named workloads: the MMA M dimension padded to 128.
    lens = [1, 90, 600]
    case = I.make_case("heads%d" % H, len(lens), 1, H, lens, seed=59)
    dc = DeviceCase(case)
    st = dc.step(num_splits=2)
    check_case(dc, st, range(case.B), expanded_heads=[0, H - 1])


def test_block_table_out_of_range_is_flagged():
    lens = [130]
    case = I.make_case("badpage", 1, 1, 16, lens, paged=True, seed=13)
    dc = DeviceCase(case)
    dc.block_table[0, 1] = 10_000          # a page id outside the pool
    st = dc.step(num_splits=1)
    import mla_latent_kv_70_b300 as mla
    assert int(st.status.item()) & mla.FLAG_BLOCK_TABLE
    assert np.all(np.isfinite(st.o_lat.cpu().numpy()))


# ----------------------------------------------------------------------------
# The stand-alone calls
# ----------------------------------------------------------------------------

def test_rope_inplace_matches_oracle():
    import mla_latent_kv_70_b300 as mla
    rows = 1000
    x = I.randn_bf16((rows, 576), 0, "ropetest")
    pos = torch.randint(0, 131072, (rows,), generator=torch.Generator().manual_seed(1),
                        dtype=torch.int32)
    xd = x.cuda()
    mla.mla_rope_inplace(xd, 576, rows, 512, pos.cuda(), 10000.0)
    got = xd.cpu().double().numpy()
    ref = O.rope_interleaved(x[:, 512:].double().numpy(), pos.double().numpy(), 10000.0)
    np.testing.assert_array_equal(got[:, :512], x[:, :512].double().numpy())
    # fp32 rotation stored as bf16: within two bf16 ulps of the exact value
    np.testing.assert_allclose(got[:, 512:], ref, rtol=2 ** -7, atol=2 ** -7)


def test_combine_matches_oracle():
    import mla_latent_kv_70_b300 as mla
    g = torch.Generator().manual_seed(2)
    K, rows = 7, 300
    o_part = torch.randn(K, rows, 512, generator=g)
    lse_part = torch.randn(K, rows, generator=g) * 3
    lse_part[2, :50] = -math.inf
    lse_part[:, 299] = -math.inf
    o = torch.empty(rows, 512, device="cuda")
    lse = torch.empty(rows, device="cuda")
    mla.mla_combine_partials(o_part.cuda(), lse_part.cuda(), o, lse)
    r_o, r_lse = O.combine_partials(o_part.double().numpy(), lse_part.double().numpy())
    np.testing.assert_allclose(o.cpu().numpy(), r_o, rtol=1e-5, atol=1e-5)
    assert lse_err(lse.cpu().numpy(), r_lse) < 1e-5


@pytest.mark.parametrize("B,S,H", [(3, 2, 128), (67, 2, 128), (130, 1, 16), (64, 1, 128),
                                   (128, 2, 128), (150, 2, 32)])
def test_absorb_and_out_proj_match_oracle(B, S, H):
    # M = B*S query rows per head: a few rows, ragged tiles (134, 130 rows), the
    # DeepSeek-V3 decode batch (64), the two-token batch (256: the largest single tile of
    # the absorption) and more rows than one tile (300).
    import mla_latent_kv_70_b300 as mla
    case = I.make_case("proj", B, S, H, [10] * B, seed=17)
    qn, qr = I.queries(case)
    w_uk, w_uv = I.weights(case)
    q_cat = torch.empty(B, S, H, 576, dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_q(qn.cuda(), qr.cuda(), w_uk.cuda(), None, 1e4, q_cat)
    ref = O.absorb_q(qn.double().numpy(), w_uk.double().numpy())
    got = q_cat.cpu().double().numpy()
    assert row_rel_err(got[..., :512], ref) < 1e-2
    # bf16 output of an fp32 sum: within one bf16 rounding (unit roundoff 2^-8) of the
    # exact value, plus the fp32 accumulation error over 128 terms (< 2^-16 sum |q w|).
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -16 * O.absorb_q(np.abs(qn.double().numpy()),
                                                               np.abs(w_uk.double().numpy()))
    assert np.all(np.abs(got[..., :512] - ref) <= bound)
    np.testing.assert_array_equal(got[..., 512:], qr.double().numpy())
    o_lat = torch.randn(B, S, H, 512, generator=torch.Generator().manual_seed(3))
    o = torch.empty(B, S, H, 128, device="cuda")
    mla.mla_out_proj_uv(o_lat.cuda(), w_uv.cuda(), o)
    lat, w = o_lat.double().numpy(), w_uv.double().numpy()
    r = O.out_proj_uv(lat, w)
    got = o.cpu().numpy()
    assert row_rel_err(got, r) <= ROW_REL_TOL
    # The tensor core takes o_lat rounded to bf16 (unit roundoff 2^-8: 8 significant
    # bits), accumulating in fp32: each output moves by at most 2^-8 sum_i |o_lat_i w_i|;
    # the test allows twice that.
    bound = 2.0 ** -7 * O.out_proj_uv(np.abs(lat), np.abs(w))
    assert np.all(np.abs(got - r) <= bound + 1e-6)


# ----------------------------------------------------------------------------
# The named workloads at full size (sampled sequences)
# ----------------------------------------------------------------------------

def test_dsv3_decode_full_size():
    case = I.dsv3()
    dc = DeviceCase(case)
    st = dc.step()
    check_case(dc, st, [0, 31, 63], expanded_heads=[0, 64, 127])


def test_ragged_paged_full_size():
    case = I.ragged_paged()
    dc = DeviceCase(case)
    st = dc.step()
    lens = case.seqlens
    seqs = [int(np.argmin(lens)), int(np.argmax(lens)), 7]
    check_case(dc, st, seqs, expanded_heads=[5])
    st_plan = dc.step(planned=True)              # the count planned from the lengths (8)
    assert st_plan.num_splits != st.num_splits
    check_case(dc, st_plan, seqs)


def test_long_context_splitkv_full_size():
    case = I.long_splitkv(num_splits=64)
    dc = DeviceCase(case)
    st = dc.step()
    check_case(dc, st, [0, 1], expanded_heads=[1])
    st_auto = dc.step(num_splits=0)
    check_case(dc, st_auto, [0, 1])


def test_mtp_causal_full_size():
    case = I.mtp()
    dc = DeviceCase(case)
    st = dc.step()
    check_case(dc, st, [0, 64, 127], expanded_heads=[3])
    st_plan = dc.step(planned=True)              # planned from the lengths: one split
    assert st_plan.num_splits == 1
    check_case(dc, st_plan, [0, 127])


# ----------------------------------------------------------------------------
# Ordering between the kernels of consecutive steps, and split planning
# ----------------------------------------------------------------------------

def test_back_to_back_steps_see_their_own_inputs():
    # Each kernel of a step may start before the previous kernel ends (programmatic
    # dependent launch) and waits for it only before touching shared buffers.  Two steps
    # issued without a host synchronisation, on the same buffers, with different queries,
    # must each match the oracle; the first step's outputs are copied out between them
    # on the stream.
    case = I.make_case("b2b", 4, 1, 128, [700, 64, 1900, 5], seed=31)
    dc = DeviceCase(case)
    import mla_latent_kv_70_b300 as mla
    st = mla.DecodeStep(case.B, case.S, case.H, dc.w_uk, dc.w_uv, max_seqlen=max(case.seqlens),
                        num_splits=3)
    case2 = I.make_case("b2b", 4, 1, 128, [700, 64, 1900, 5], seed=32)
    qn2, qr2 = (t.cuda() for t in I.queries(case2))
    st(dc.q_nope, dc.q_rope, dc.kv, dc.seqlens)
    o1, lse1 = st.o.clone(), st.lse.clone()
    st(qn2, qr2, dc.kv, dc.seqlens)
    torch.cuda.synchronize()
    w_uk, w_uv = (w.double().numpy() for w in I.weights(case))
    for b in range(case.B):
        _, r_lse, r_o = oracle_seq(case, b, w_uk, w_uv)
        assert row_rel_err(o1[b].cpu().numpy(), r_o) <= ROW_REL_TOL
        check_lse(lse1[b].cpu().numpy(), r_lse, lse_tolerance(case, b, w_uk), where=b)
        # the second step: same cache, the queries of seed 32
        T = case.seqlens[b]
        rows = I.seq_rows(case, b)[:T].double().numpy()
        q_lat = O.absorb_q(I.seq_queries(case2, b)[0].double().numpy(), w_uk)
        o_lat, lse = O.decode_absorbed_seq(q_lat, I.seq_queries(case2, b)[1].double().numpy(),
                                           rows[:, :512], rows[:, 512:], case.scale)
        assert row_rel_err(st.o[b].cpu().numpy(), O.out_proj_uv(o_lat, w_uv)) <= ROW_REL_TOL


@pytest.mark.parametrize("splits", [5, 128])
def test_mostly_empty_splits(splits):
    # Splits are chunks of ceil(max_seqlen / splits) rows for every sequence: with a short
    # and a long sequence most of the short one's splits are empty and exit at once.
    lens = [3, 4000]
    case = I.make_case("empty_splits", 2, 1, 128, lens, seed=33)
    dc = DeviceCase(case)
    st = dc.step(num_splits=splits)
    check_case(dc, st, range(case.B))
