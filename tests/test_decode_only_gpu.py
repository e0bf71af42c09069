"""GPU parity of the latent decode on its own (mla_decode_latent through the C ABI).

The queries are seeded q_cat rows ([q~ | q^R], bf16) rather than the output of the key
absorption, so the kernel and the oracle read identical query values: the comparison then
measures the decode's own arithmetic (fp32 scores, the fp16 exchange of the peer CTA's
half of each score, bf16 P for the tensor core, the online softmax and the split merge),
and every lse is held to 1e-3 absolute however short the sequence.  The shapes cover
every shape the C ABI accepts: 1 to 4 query tokens (causal), head counts 16 to 128 in
steps of 16, contiguous and paged caches, 1 to 128 splits, empty and one-row sequences.
"""
import numpy as np
import pytest
import torch

from mla_latent_kv_70_b300 import inputs as I
from tests.mla_cases import DecodeOnlyCase, check_decode_only

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_70_b300 import build
    build.build()


def nan_tail(dc: DecodeOnlyCase):
    """Rows past each sequence's end hold NaN: the kernel must never use them."""
    case = dc.case
    for b, T in enumerate(case.seqlens):
        if case.paged:
            n = case.pages_per_seq[b]
            last = int(case.block_table[b, n - 1])
            dc.kv[last, T - (n - 1) * 64:] = float("nan")
        else:
            dc.kv[b, T:] = float("nan")


@pytest.mark.parametrize("H", [16, 48, 112, 128])
@pytest.mark.parametrize("splits", [1, 3, 64])
def test_short_and_ragged_lengths(H, splits):
    lens = [1, 2, 5, 63, 64, 65, 0, 129, 200]
    case = I.make_case("dec_edges", len(lens), 1, H, lens, t_cap=256, seed=41)
    dc = DecodeOnlyCase(case)
    nan_tail(dc)
    o_lat, lse = dc.run(num_splits=splits, max_seqlen=256)
    check_decode_only(case, o_lat, lse, range(case.B))
    assert np.all(o_lat[6] == 0) and np.all(np.isneginf(lse[6]))


@pytest.mark.parametrize("splits", [1, 2])
def test_every_tile_count_up_to_13(splits):
    # One sequence per tile count 1..13, each with a ragged last tile: every residue of
    # the kernel's barrier cycles (period 6 tiles) appears twice.
    lens = [64 * n - (7 * n) % 64 for n in range(1, 14)]
    case = I.make_case("dec_tiles", len(lens), 1, 128, lens, t_cap=13 * 64, seed=43)
    dc = DecodeOnlyCase(case)
    nan_tail(dc)
    o_lat, lse = dc.run(num_splits=splits, max_seqlen=13 * 64)
    check_decode_only(case, o_lat, lse, range(case.B))


@pytest.mark.parametrize("S", [2, 3, 4])
@pytest.mark.parametrize("H", [32, 128])
@pytest.mark.parametrize("splits", [1, 3])
def test_causal_query_tokens(S, H, splits):
    # S query tokens per sequence are its last S rows; token s reads rows j <= T-S+s.
    lens = [S, S + 1, 7, 100, 300]
    case = I.make_case("dec_causal", len(lens), S, H, lens, causal=True, seed=45 + S)
    dc = DecodeOnlyCase(case)
    nan_tail(dc)
    o_lat, lse = dc.run(num_splits=splits)
    check_decode_only(case, o_lat, lse, range(case.B))


@pytest.mark.parametrize("causal,S", [(False, 1), (True, 2), (True, 4)])
@pytest.mark.parametrize("splits", [1, 4])
def test_paged(causal, S, splits):
    lens = [70, 1, 300, 64, 2]
    case = I.make_case("dec_paged", len(lens), S, 128, lens, paged=True, causal=causal, seed=47)
    dc = DecodeOnlyCase(case)
    nan_tail(dc)
    o_lat, lse = dc.run(num_splits=splits)
    check_decode_only(case, o_lat, lse, range(case.B))


@pytest.mark.parametrize("splits", [5, 128])
def test_mostly_empty_splits(splits):
    lens = [3, 4000]
    case = I.make_case("dec_empty_splits", 2, 1, 128, lens, seed=49)
    dc = DecodeOnlyCase(case)
    o_lat, lse = dc.run(num_splits=splits)
    check_decode_only(case, o_lat, lse, range(case.B))


def test_dsv3_decode_full_size_sampled():
    # The DeepSeek-V3-shaped decode in the bench's launch configuration, sampled.
    case = I.dsv3()
    dc = DecodeOnlyCase(case)
    o_lat, lse = dc.run()
    check_decode_only(case, o_lat, lse, [0, 17, 63])
