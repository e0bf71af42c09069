"""FP8 latent cache ("DeepSeek Multi-Head Latent Attention(MLA) 아키텍처 해부", section 5, the
checklist item on FP8 mixed precision): the quantizer against the oracle byte for byte,
and the decode over the FP8 form against the oracle's attention over the dequantized
rows (o_lat rows within 1e-2, LSE within 1e-3), plus the host-side rejects.

The decode's inputs are drawn directly in the FP8 form (inputs.seq_fp8_rows: codes and
power-of-two scales from a seeded generator), so the oracle's inputs never pass through
the CUDA quantizer."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from mla_latent_kv_70_b300 import inputs as I
from tests.mla_cases import LSE_ABS_TOL, ROW_REL_TOL, check_lse, log_lse, lse_err, rounding_lse_tol, row_rel_err

P = 4096  # a fake 16-byte aligned address: a call rejected on the host never dereferences it


@pytest.fixture(scope="module")
def lib():
    import mla_latent_kv_70_b300 as mla
    from mla_latent_kv_70_b300 import build
    build.build()
    return mla.lib()


# ----------------------------------------------------------------------------
# Host-side rejects (no GPU)
# ----------------------------------------------------------------------------

def test_quantize_rejects_on_the_host(lib):
    f = lib.mla_quantize_fp8
    assert f(None, 576, 4, P, P, None) == 1
    assert f(P, 576, 4, None, P, None) == 1
    assert f(P, 576, 4, P, None, None) == 1
    assert f(P, 570, 4, P, P, None) == 1          # row stride below 576
    assert f(P, 580, 4, P, P, None) == 1          # row stride not a multiple of 8
    assert f(P + 8, 576, 4, P, P, None) == 1      # rows not 16-byte aligned
    assert f(P, 576, 4, P + 4, P, None) == 1      # kv8 not 16-byte aligned
    assert f(P, 576, 4, P, P + 2, None) == 1      # scales not 4-byte aligned
    assert f(P, 576, -1, P, P, None) == 1
    assert f(P, 576, 0, P, P, None) == 0          # nothing to do


def fp8_args(**over):
    a = dict(q_cat=P, kv8=P, kv_scale=P, kv_seq_stride=256, seqlens=P, block_table=None, max_pages=0,
             page_size=64, num_pages=0, B=4, S=1, H=16, causal=0, scale=0.07, num_splits=1,
             max_seqlen=256, o_lat=P, lse=P, workspace=None, workspace_bytes=0, status=None, stream=None)
    a.update(over)
    return list(a.values())


@pytest.mark.parametrize("over,code", [
    (dict(kv_scale=None), 1), (dict(kv_scale=P + 4), 1), (dict(kv_seq_stride=258, max_seqlen=256), 1),
    (dict(kv8=None), 1), (dict(kv8=P + 8), 1),
    (dict(q_cat=None), 1), (dict(H=24), 2), (dict(S=5), 2), (dict(num_splits=129), 1),
    (dict(block_table=P, page_size=32, max_pages=4, num_pages=4), 2)])
def test_decode_fp8_rejects_on_the_host(lib, over, code):
    assert lib.mla_decode_latent_fp8(*fp8_args(**over)) == code


# ----------------------------------------------------------------------------
# Quantizer: bit for bit
# ----------------------------------------------------------------------------

@pytest.mark.gpu
def test_quantize_matches_the_oracle_bytewise(lib):
    import mla_latent_kv_70_b300 as mla
    g = torch.Generator().manual_seed(11)
    n = 1500
    x = torch.randn(n, I.ROW, generator=g) * torch.pow(10.0, torch.empty(n, 1).uniform_(-3, 3, generator=g))
    x[0] = 0.0                                               # all-zero row: scale 1
    x[1, 7] = 3.0e6                                          # one large value
    x[2, :I.D_C] = 1e9                                       # beyond 448 * 2^15: saturates
    x[3, :I.D_C] = torch.randn(I.D_C, generator=g) * 1e-38   # bf16 subnormals
    ties = torch.tensor([448.0, 1.0625, 1.1875, -1.0625, 2.0 ** -10, 1.5 * 2.0 ** -10, -2.0 ** -11, 0.0])
    x[4, :ties.numel()] = ties                               # scale 1: exact ties and tiny values
    x[4, ties.numel():I.D_C] = 0.5
    rows = torch.zeros(n, I.ROW + 8, dtype=torch.bfloat16)   # a row stride of 584
    rows[:, :I.ROW] = x.to(torch.bfloat16)
    ref_codes, ref_kr, ref_scales = O.quantize_fp8_rows(rows[:, :I.ROW].double().numpy())
    d_rows = rows.cuda()
    kv8 = torch.full((n, I.FP8_ROW), 0xAA, dtype=torch.uint8, device="cuda")
    sc = torch.full((n,), float("nan"), device="cuda")
    mla.mla_quantize_fp8(d_rows[:, :I.ROW], kv8, sc)
    torch.cuda.synchronize()
    kv8, sc = kv8.cpu().numpy(), sc.cpu().numpy()
    mism = np.argwhere(kv8[:, :I.D_C] != ref_codes)
    assert mism.size == 0, (mism[:5], kv8[tuple(mism[0])], ref_codes[tuple(mism[0])])
    assert np.array_equal(kv8[:, I.D_C:], rows[:, I.D_C:I.ROW].contiguous().view(torch.uint8).numpy())
    assert np.array_equal(sc.astype(np.float64), ref_scales)


# ----------------------------------------------------------------------------
# Decode over the FP8 form
# ----------------------------------------------------------------------------

class Fp8Case:
    def __init__(self, case):
        self.case = case
        self.kv8, self.sc = I.fp8_cache(case, device="cuda")
        if not case.paged:   # rows past each sequence hold NaN codes and NaN scales
            for b, T in enumerate(case.seqlens):
                self.kv8[b, T:, :I.D_C] = 0x7F
                self.sc[b, T:] = float("nan")
        self.q_cat = I.q_cat(case).cuda()
        self.seqlens = torch.tensor(case.seqlens, dtype=torch.int32, device="cuda")
        self.block_table = case.block_table.cuda() if case.paged else None

    def run(self, num_splits):
        import mla_latent_kv_70_b300 as mla
        c = self.case
        T = max(c.seqlens)
        o_lat = torch.full((c.B, c.S, c.H, I.D_C), float("nan"), device="cuda")
        lse = torch.full((c.B, c.S, c.H), float("nan"), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = mla.mla_decode_workspace_bytes(c.B, c.S, c.H, num_splits, T)
        ws = torch.empty(ws // 4, device="cuda") if ws else None
        mla.mla_decode_latent_fp8(self.q_cat, self.kv8, self.sc, self.seqlens, o_lat, lse, scale=c.scale,
                                  max_seqlen=T, block_table=self.block_table, causal=c.causal,
                                  num_splits=num_splits, workspace=ws, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        return o_lat.cpu().numpy(), lse.cpu().numpy()


def oracle_fp8_seq(case, b):
    """The oracle's attention of sequence b over its dequantized FP8 rows."""
    T = case.seqlens[b]
    rows, sc = I.seq_fp8_rows(case, b)
    rows, sc = rows[:T], sc[:T]
    kr = rows[:, I.D_C:].contiguous().view(torch.bfloat16).double().numpy()
    cache = O.dequantize_fp8_rows(rows[:, :I.D_C].numpy(), kr, sc.double().numpy())
    q = I.seq_q_cat(case, b).double().numpy()
    return O.decode_absorbed_seq(q[..., :I.D_C], q[..., I.D_C:], cache[:, :I.D_C], cache[:, I.D_C:],
                                 case.scale, case.causal)


def check_fp8(case, o_lat, lse, seqs, key):
    for b in seqs:
        r_lat, r_lse = oracle_fp8_seq(case, b)
        assert row_rel_err(o_lat[b], r_lat) <= ROW_REL_TOL, (key, b)
        err = lse_err(lse[b], r_lse)
        log_lse(key, err, LSE_ABS_TOL)
        assert err <= LSE_ABS_TOL, (key, b, err)


CASES = {
    # every tile count 1..11 with ragged tails, T = 1 and an empty sequence
    "ragged": lambda: I.make_case("fp8_ragged", 5, 1, 16, [1, 0, 200, 700, 64], seed=21, t_cap=720),
    "heads128": lambda: I.make_case("fp8_h128", 2, 1, 128, [333, 1024], seed=22, t_cap=1040),
    "causal_s2": lambda: I.make_case("fp8_causal", 3, 2, 64, [2, 130, 511], causal=True, seed=23, t_cap=520),
    "paged": lambda: I.make_case("fp8_paged", 3, 1, 32, [64, 640, 1000], paged=True, seed=24),
    "paged_causal_s3": lambda: I.make_case("fp8_paged_c3", 2, 3, 16, [5, 900], paged=True, causal=True, seed=25),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("splits", [1, 3])
def test_decode_fp8_matches_the_oracle(lib, name, splits):
    case = CASES[name]()
    fc = Fp8Case(case)
    o_lat, lse = fc.run(splits)
    check_fp8(case, o_lat, lse, range(case.B), f"{name}/{splits}")


@pytest.mark.gpu
def test_decode_fp8_equals_the_bf16_decode_on_the_widened_cache(lib):
    # Widening E4M3 * (power-of-two scale) to bf16 is exact, so the bf16 decode over the
    # widened rows reads the same operands in the same order: the results agree bit for bit.
    import mla_latent_kv_70_b300 as mla
    case = I.make_case("fp8_same", 4, 1, 128, [1, 100, 1000, 2048], seed=26, t_cap=2048)
    fc = Fp8Case(case)
    codes = fc.kv8[..., :I.D_C].contiguous().view(torch.float8_e4m3fn).float()
    lat = torch.nan_to_num(codes * fc.sc[..., None], nan=0.0)
    kv = torch.cat([lat.to(torch.bfloat16), fc.kv8[..., I.D_C:].contiguous().view(torch.bfloat16)], dim=-1)
    for splits in (1, 2):
        o8, l8 = fc.run(splits)
        o = torch.empty(case.B, 1, case.H, I.D_C, device="cuda")
        l = torch.empty(case.B, 1, case.H, device="cuda")
        ws = mla.mla_decode_workspace_bytes(case.B, 1, case.H, splits, 2048)
        ws = torch.empty(ws // 4, device="cuda") if ws else None
        mla.mla_decode_latent(fc.q_cat, kv.contiguous(), fc.seqlens, o, l, scale=case.scale, max_seqlen=2048,
                              num_splits=splits, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(o.cpu().numpy(), o8) and np.array_equal(l.cpu().numpy(), l8), splits


@pytest.mark.gpu
def test_decode_fp8_deepseek_v3_full_size(lib):
    case = I.make_case("fp8_dsv3", 64, 1, 128, [4096] * 64, seed=27)
    fc = Fp8Case(case)
    o_lat, lse = fc.run(1)
    check_fp8(case, o_lat, lse, [0, 31, 63], "dsv3_fp8")


@pytest.mark.gpu
@pytest.mark.parametrize("splits", [1, 3])
def test_decode_fp8_timeout_is_flagged_and_device_recovers(lib, splits):
    # The test hook withholds the score commit of each unit's first tile and shortens the
    # wait limit to 1 ms: every unit gives up, records the timeout and writes the empty
    # result; the next ordinary call on the same device matches the oracle.
    import mla_latent_kv_70_b300 as mla
    case = I.make_case("fp8_timeout", 3, 1, 128, [300, 130, 64], seed=62, t_cap=320)
    fc = Fp8Case(case)
    o_lat = torch.full((case.B, 1, case.H, I.D_C), float("nan"), device="cuda")
    lse = torch.full((case.B, 1, case.H), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = mla.mla_decode_workspace_bytes(case.B, 1, case.H, splits, 300)
    ws = torch.empty(ws // 4, device="cuda") if ws else None
    mla.mla_debug_inject_timeout(mla.FAULT_DECODE, 1.0)
    try:
        mla.mla_decode_latent_fp8(fc.q_cat, fc.kv8, fc.sc, fc.seqlens, o_lat, lse, scale=case.scale,
                                  max_seqlen=300, num_splits=splits, workspace=ws, status=status)
        torch.cuda.synchronize()
    finally:
        mla.mla_debug_inject_timeout(0)
    assert int(status.item()) & mla.FLAG_TIMEOUT
    assert torch.all(o_lat == 0) and torch.all(torch.isneginf(lse))
    o_lat, lse = fc.run(splits)
    check_fp8(case, o_lat, lse, range(case.B), f"fp8_recovery/{splits}")


# ----------------------------------------------------------------------------
# Append into the FP8 cache
# ----------------------------------------------------------------------------

def test_append_fp8_rejects_on_the_host(lib):
    f = lib.mla_append_latent_fp8
    ok = dict(rows=P, B=2, S=1, theta=1e4, seqlens=P, kv8=P, sc=P, stride=64, bt=None, max_pages=0,
              page_size=64, num_pages=0, status=None, stream=None)
    call = lambda **o: f(*{**ok, **o}.values())
    assert call(rows=None) == 1 and call(kv8=None) == 1 and call(sc=None) == 1
    assert call(S=5) == 1 and call(theta=-1.0) == 1 and call(kv8=P + 8) == 1 and call(sc=P + 2) == 1
    assert call(bt=P, max_pages=2, num_pages=4, page_size=32) == 2


@pytest.mark.gpu
@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("S,theta", [(1, 10000.0), (3, 0.0)])
def test_append_fp8_places_quantized_rows(lib, paged, S, theta):
    import mla_latent_kv_70_b300 as mla
    lens = [5, 0, 100, 63]
    case = I.make_case("append8", len(lens), S, 16, [T + S for T in lens], paged=paged, seed=81, t_cap=128)
    kv8, sc = I.fp8_cache(case, device="cuda")
    before8, before_sc = kv8.cpu(), sc.cpu()
    new = torch.stack([I.randn_bf16((S, I.ROW), case.seed, "new8", b) for b in range(case.B)])
    new[0, 0, :I.D_C] = 0.0                         # an all-zero latent row: scale 1
    seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = case.block_table.cuda() if paged else None
    mla.mla_append_latent_fp8(new.cuda(), seqlens, kv8, sc, rope_theta=theta, block_table=bt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert seqlens.cpu().tolist() == [T + S for T in lens]
    after8, after_sc = kv8.cpu(), sc.cpu()
    written = torch.zeros(after8.shape[:-1], dtype=torch.bool)
    for b, T in enumerate(lens):
        rows = new[b].double().numpy()
        codes, _, scales = O.quantize_fp8_rows(rows)
        ref, pos = O.append_latent_rows(rows, T, theta or None)
        for s, t in enumerate(pos):
            t = int(t)
            if paged:
                page = int(case.block_table[b, t // 64])
                got8, got_sc = after8[page, t % 64], after_sc[page, t % 64]
                written[page, t % 64] = True
            else:
                got8, got_sc = after8[b, t], after_sc[b, t]
                written[b, t] = True
            np.testing.assert_array_equal(got8[:I.D_C].numpy(), codes[s])          # codes: byte for byte
            assert float(got_sc) == scales[s]
            kr = got8[I.D_C:].contiguous().view(torch.bfloat16).double().numpy()
            np.testing.assert_allclose(kr, ref[s, I.D_C:], rtol=2 ** -7, atol=2 ** -7)   # k^R rotated, bf16
    assert torch.equal(after8[~written], before8[~written])
    assert torch.equal(after_sc[~written], before_sc[~written])


@pytest.mark.gpu
def test_fp8_step_that_appends_matches_the_oracle(lib):
    # A DecodeStep over the FP8 cache that appends its token's row first: the decode then
    # reads the quantized new row at its position.
    import mla_latent_kv_70_b300 as mla
    lens = [63, 200, 1]
    case = I.make_case("fp8_step", 3, 1, 32, [T + 1 for T in lens], seed=83, t_cap=256)
    kv8, sc = I.fp8_cache(case, device="cuda")
    new = torch.stack([I.randn_bf16((1, I.ROW), case.seed, "new8s", b) for b in range(case.B)])
    qn, qr = I.queries(case)
    w_uk, w_uv = I.weights(case)
    seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    step = mla.DecodeStep(case.B, 1, case.H, w_uk.cuda(), w_uv.cuda(), max_seqlen=max(lens) + 1, num_splits=2)
    step(qn.cuda(), qr.cuda(), kv8, seqlens, new_rows=new.cuda(), kv_scale=sc)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    o_lat, lse = step.o_lat.cpu().numpy(), step.lse.cpu().numpy()
    wk = w_uk.double().numpy()
    for b, T in enumerate(lens):
        rows, s_ = I.seq_fp8_rows(case, b)
        kr = rows[:T, I.D_C:].contiguous().view(torch.bfloat16).double().numpy()
        cache = O.dequantize_fp8_rows(rows[:T, :I.D_C].numpy(), kr, s_[:T].double().numpy())
        codes, nkr, nsc = O.quantize_fp8_rows(new[b].double().numpy())
        cache = np.concatenate([cache, O.dequantize_fp8_rows(codes, nkr, nsc)])
        q_lat = O.absorb_q(qn[b].double().numpy(), wk)
        r_lat, r_lse = O.decode_absorbed_seq(q_lat, qr[b].double().numpy(), cache[:, :I.D_C], cache[:, I.D_C:],
                                             case.scale)
        assert row_rel_err(o_lat[b], r_lat) <= ROW_REL_TOL, b
        # q~ is stored in bf16 on the GPU and exact in the oracle: the derived bound of the
        # absorb -> decode path (every sequence here reads fewer than 256 rows)
        tol = rounding_lse_tol(q_lat[0], qr[b].double().numpy()[0], cache[:, :I.D_C], cache[:, I.D_C:], case.scale)
        check_lse(lse[b][0], r_lse[0], tol, key="fp8_step", where=b)
