"""The seeded synthetic workloads (mla_latent_kv_70_b300/inputs.py): reproducible, with the
shapes and structure the measurements state, and a valid page table."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from mla_latent_kv_70_b300 import inputs as I  # noqa: E402


def test_same_seed_same_data_other_seed_other_data():
    a, b, c = I.make_case("t", 2, 1, 16, [70, 5], seed=4), I.make_case("t", 2, 1, 16, [70, 5], seed=4), \
        I.make_case("t", 2, 1, 16, [70, 5], seed=5)
    assert torch.equal(I.cache(a), I.cache(b)) and not torch.equal(I.cache(a), I.cache(c))
    for x, y in zip(I.queries(a) + I.weights(a), I.queries(b) + I.weights(b)):
        assert torch.equal(x, y)


def test_workload_shapes():
    d = I.dsv3()
    assert (d.B, d.S, d.H, d.total_tokens) == (64, 1, 128, 64 * 4096)
    qn, qr = I.queries(d)
    assert qn.shape == (64, 1, 128, 128) and qr.shape == (64, 1, 128, 64)
    assert qn.dtype == qr.dtype == torch.bfloat16
    w_uk, w_uv = I.weights(d)
    assert w_uk.shape == w_uv.shape == (128, 512, 128)
    m = I.mtp()
    assert (m.B, m.S, m.causal, m.rope) == (128, 2, True, True)
    assert m.q_positions()[0].tolist() == [8190, 8191]    # the last two rows of the sequence
    lc = I.long_splitkv()
    assert lc.seqlens == [131072, 131072]


def test_ragged_lengths_and_page_table():
    r = I.ragged_paged()
    assert r.B == 32 and all(512 <= t <= 32768 for t in r.seqlens)
    assert r.seqlens == I.ragged_paged().seqlens              # seeded
    assert r.pages_per_seq == [-(-t // 64) for t in r.seqlens]
    used = torch.cat([r.block_table[b, :n] for b, n in enumerate(r.pages_per_seq)])
    # every page of the pool is used exactly once (a seeded permutation)
    assert sorted(used.tolist()) == list(range(r.num_pages))
    assert r.block_table.dtype == torch.int32


def test_weight_scale():
    w_uk, _ = I.weights(I.make_case("w", 1, 1, 16, [1], seed=0))
    std = float(w_uk.float().std())
    assert abs(std / 512 ** -0.5 - 1) < 0.1        # N(0, 1/sqrt(512)), within 10%
