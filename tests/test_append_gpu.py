"""GPU parity of the cache append (mla_append_latent through the C ABI), and of a decode
step that appends its tokens' rows before attending, against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from mla_latent_kv_70_b300 import inputs as I
from tests.mla_cases import DeviceCase, check_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_70_b300 import build
    build.build()


def stored_row(case, kv_cpu, b, t):
    """Row at position t of sequence b, read back from the cache (either layout)."""
    if case.paged:
        page = int(case.block_table[b, t // 64])
        return kv_cpu[page, t % 64]
    return kv_cpu[b, t]


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("S,theta", [(1, 10000.0), (2, 10000.0), (3, 0.0)])
def test_append_places_rows_and_rotates_k_rope(paged, S, theta):
    import mla_latent_kv_70_b300 as mla
    lens = [5, 0, 100, 63]
    case = I.make_case("append", len(lens), S, 16, [T + S for T in lens], paged=paged, seed=71,
                       t_cap=128)
    kv = I.cache(case, device="cuda")
    before = kv.cpu()
    new = torch.stack([I.randn_bf16((S, 576), case.seed, "new", b) for b in range(case.B)]).cuda()
    seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = case.block_table.cuda() if paged else None
    mla.mla_append_latent(new, seqlens, kv, rope_theta=theta, block_table=bt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert seqlens.cpu().tolist() == [T + S for T in lens]
    after = kv.cpu()
    written = torch.zeros(after.shape[:-1], dtype=torch.bool)
    for b, T in enumerate(lens):
        ref, pos = O.append_latent_rows(new[b].cpu().double().numpy(), T, theta or None)
        for s, t in enumerate(pos):
            got = stored_row(case, after, b, int(t)).double().numpy()
            np.testing.assert_array_equal(got[:512], ref[s, :512])     # c^KV: bit for bit
            # k^R: fp32 rotation stored as bf16, within two bf16 ulps of the exact value
            np.testing.assert_allclose(got[512:], ref[s, 512:], rtol=2 ** -7, atol=2 ** -7)
            if paged:
                written[int(case.block_table[b, t // 64]), t % 64] = True
            else:
                written[b, t] = True
    assert torch.equal(after[~written], before[~written])             # nothing else moved


def test_append_out_of_place_rows_are_flagged_and_skipped():
    import mla_latent_kv_70_b300 as mla
    lens = [62, 10]
    case = I.make_case("append_bad", 2, 4, 16, [66, 14], paged=True, seed=73)
    kv = I.cache(case, device="cuda")
    before = kv.clone()
    bt = case.block_table.clone()
    bt[0, 1] = 10_000                      # rows 64, 65 of sequence 0 have no page
    new = torch.stack([I.randn_bf16((4, 576), case.seed, "new", b) for b in range(2)]).cuda()
    seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_append_latent(new, seqlens, kv, rope_theta=1e4, block_table=bt.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mla.FLAG_BLOCK_TABLE
    assert seqlens.cpu().tolist() == [66, 14]
    page0 = int(case.block_table[0, 0])
    assert torch.equal(kv[page0, :62], before[page0, :62])
    assert not torch.equal(kv[page0, 62:64], before[page0, 62:64])    # the rows with a place


@pytest.mark.parametrize("paged", [False, True])
def test_decode_step_after_append_matches_oracle(paged):
    # The cache holds T - S rows of each sequence; the step appends the last S rows (k^R
    # rotated on the way in) and then attends causally: the result must be the oracle's
    # attention over all T rows.
    import mla_latent_kv_70_b300 as mla
    lens = [300, 2, 1500]
    S = 2
    case = I.make_case("append_step", len(lens), S, 128, lens, paged=paged, causal=True, rope=True,
                       seed=75)
    dc = DeviceCase(case)                  # every cached row rotated in place
    for b, T in enumerate(lens):           # forget the last S rows of each sequence
        for t in range(T - S, T):
            if paged:
                dc.kv[int(case.block_table[b, t // 64]), t % 64] = float("nan")
            else:
                dc.kv[b, t] = float("nan")
    dc.seqlens -= S
    new = torch.stack([I.seq_rows(case, b)[T - S:T] for b, T in enumerate(lens)]).cuda()
    mla.mla_append_latent(new, dc.seqlens, dc.kv, rope_theta=case.theta, block_table=dc.block_table)
    assert dc.seqlens.cpu().tolist() == lens
    st = dc.step(num_splits=1)
    check_case(dc, st, range(case.B), expanded_heads=[7])


def test_decode_step_with_append_replays_as_a_graph():
    # DecodeStep(new_rows=...) runs append -> absorb -> decode -> W_UV; captured as a CUDA
    # graph and replayed after the cache and seqlens are put back, it gives the oracle.
    import mla_latent_kv_70_b300 as mla
    lens = [700, 65]
    S = 2
    case = I.make_case("append_graph", len(lens), S, 128, lens, causal=True, rope=True, seed=77)
    dc = DeviceCase(case)
    for b, T in enumerate(lens):
        dc.kv[b, T - S:T] = float("nan")
    start = torch.tensor([T - S for T in lens], dtype=torch.int32, device="cuda")
    dc.seqlens.copy_(start)
    new = torch.stack([I.seq_rows(case, b)[T - S:T] for b, T in enumerate(lens)]).cuda()
    st = mla.DecodeStep(case.B, S, case.H, dc.w_uk, dc.w_uv, max_seqlen=max(lens), num_splits=2,
                        causal=True, rope_theta=case.theta, rope=True)
    replay = st.capture(dc.q_nope, dc.q_rope, dc.kv, dc.seqlens, q_pos=dc.q_pos, new_rows=new)
    torch.cuda.synchronize()
    for b, T in enumerate(lens):
        dc.kv[b, T - S:T] = float("nan")
    dc.seqlens.copy_(start)
    replay()
    torch.cuda.synchronize()
    assert dc.seqlens.cpu().tolist() == lens
    check_case(dc, st, range(case.B))
