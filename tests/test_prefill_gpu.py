"""GPU parity of prefill / chunked prefill (mla_prefill through the C ABI) against the
oracle's expanded definition: per-head K_h = C W_UK[h], V_h = C W_UV[h], causal softmax
attention of the last T_q positions over the first T_kv cached rows."""
import numpy as np
import pytest
import torch

import oracle as O
from mla_latent_kv_70_b300 import inputs as I
from tests.mla_cases import (K_HOEFFDING, LSE_ABS_TOL, ROW_REL_TOL, SHORT_T, U_BF16, check_lse,
                             row_rel_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_70_b300 import build
    build.build()


def prefill_lse_tolerance(qn, qr, C, KR, w_uk, scale, heads):
    """[S, len(heads)] bound on |lse_gpu - lse_exact|: LSE_ABS_TOL for query tokens that read
    at least SHORT_T rows; below that, plus the effect of storing K_h = C W_UK[h] in bf16
    (each element moves by at most 2^-8 of itself), bounded as for the decode path by
    Hoeffding's inequality over those independent roundings: first order
    sum_j a_j scale sum_d q_d e_jd, second order max_j d_j^2 / 2."""
    S, T = qn.shape[0], C.shape[0]
    tol = np.full((S, len(heads)), LSE_ABS_TOL)
    k, u = K_HOEFFDING, U_BF16
    for hi, h in enumerate(heads):
        K = C @ w_uk[h]                                     # [T, 128]
        for s in range(S):
            n = O.visible_length(T, S, s, True)
            if n >= SHORT_T:
                continue
            x = (K[:n] @ qn[s, h] + KR[:n] @ qr[s, h]) * scale
            a = np.exp(x - x.max())
            a /= a.sum()
            per = (qn[s, h] ** 2) @ (K[:n] ** 2).T            # [n]: sum_d q_d^2 K_jd^2
            first = k * scale * u * np.sqrt((a ** 2) @ per)
            second = 0.5 * (k * scale * u) ** 2 * per.max()
            tol[s, hi] = LSE_ABS_TOL + first + second
    return tol


# Query blocks of 128 rows: 300 leaves a last block of 44 queries (its other rows are never
# written); 200/200 ends the sequence inside a key tile (the rows past the end are cleared
# in the value tile); 512/600 and 600/900 are chunked prefill (the queries are the last T_q
# positions).  Blocks i and n-1-i of a head form one unit of the persistent schedule:
# 1024 with 128 heads and 600/900 with two sequences of 64 heads give each CTA several
# units, and the five blocks of 600 leave the middle one without a partner.  One query
# over 5 rows, and one over one row, are the smallest chunks.
@pytest.mark.parametrize("B,T_q,T_kv,H", [(2, 300, 300, 16), (1, 130, 700, 16), (1, 64, 64, 32),
                                          (1, 200, 1000, 128), (1, 200, 200, 16), (1, 512, 600, 16),
                                          (1, 1024, 1024, 128), (2, 600, 900, 64), (3, 1, 5, 16),
                                          (1, 1, 1, 16)])
def test_prefill_matches_oracle(B, T_q, T_kv, H):
    import mla_latent_kv_70_b300 as mla
    case = I.make_case("prefill", B, T_q, H, [T_kv] * B, causal=True, seed=91, t_cap=T_kv + 40)
    kv = I.cache(case, device="cuda")
    kv[:, T_kv:] = float("nan")                 # rows past the sequence must never be used
    qn, qr = I.queries(case)
    w_uk, w_uv = I.weights(case)
    # One batch more than asked for, holding a sentinel: the tiles of the last query block
    # must not be written past row T_q of the last sequence.
    o_all = torch.full((B + 1, T_q, H, 128), 7.0, device="cuda")
    lse_all = torch.full((B + 1, T_q, H), 7.0, device="cuda")
    o, lse = o_all[:B], lse_all[:B]
    ws = torch.empty(mla.mla_prefill_workspace_bytes(B, case.t_cap, H), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_prefill(qn.cuda(), qr.cuda(), kv, T_kv, w_uk.cuda(), w_uv.cuda(), o, lse, scale=case.scale,
                    workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bool((o_all[B] == 7.0).all()) and bool((lse_all[B] == 7.0).all())
    heads = list(range(H)) if H <= 32 else [0, H // 2 - 3, H - 1]
    wk, wv = w_uk.double().numpy(), w_uv.double().numpy()
    for b in range(B):
        rows = I.seq_rows(case, b)[:T_kv].double().numpy()
        C, KR = rows[:, :512], rows[:, 512:]
        q_n, q_r = (t.double().numpy() for t in I.seq_queries(case, b))
        r_o, r_lse = O.decode_expanded_seq(q_n[:, heads], q_r[:, heads], C, KR, wk[heads], wv[heads],
                                           case.scale, causal=True)
        assert row_rel_err(o[b][:, heads].cpu().numpy(), r_o) <= ROW_REL_TOL, b
        tol = prefill_lse_tolerance(q_n, q_r, C, KR, wk, case.scale, heads)
        check_lse(lse[b][:, heads].cpu().numpy(), r_lse, tol, where=b)


@pytest.mark.parametrize("B,T,H", [(2, 300, 16), (1, 1000, 128), (3, 129, 32)])
def test_prefill_expansion_matches_definition(B, T, H):
    """The K_h and V_h that mla_prefill leaves in its workspace (bf16 [B * kv_seq_stride][H][128],
    K_h then V_h) against K_h[t] = c_t W_UK[h], V_h[t] = c_t W_UV[h] in fp64: the result of an
    fp32 sum rounded once to bf16 (unit roundoff u = 2^-8), so |gpu - exact| <= u |exact| +
    (fp32 sum error), the latter bounded by 2^-14 sum_k |c_k w_k| (twice the worst case of 512
    fp32 roundings)."""
    import mla_latent_kv_70_b300 as mla
    case = I.make_case("prefill", B, T, H, [T] * B, causal=True, seed=93, t_cap=T + 40)
    kv = I.cache(case, device="cuda")
    kv[:, T:] = float("nan")
    qn, qr = I.queries(case)
    w_uk, w_uv = I.weights(case)
    o = torch.empty(B, T, H, 128, device="cuda")
    lse = torch.empty(B, T, H, device="cuda")
    ws = torch.empty(mla.mla_prefill_workspace_bytes(B, case.t_cap, H), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_prefill(qn.cuda(), qr.cuda(), kv, T, w_uk.cuda(), w_uv.cuda(), o, lse, scale=case.scale,
                    workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    exp = ws.view(torch.bfloat16).view(2, B, case.t_cap, H, 128).float().cpu().numpy()
    heads = list(range(H)) if H <= 32 else [0, 1, 63, 64, 126, 127]
    for which, w in enumerate((w_uk, w_uv)):
        wd = w.double().numpy()
        for b in range(B):
            C = I.seq_rows(case, b)[:T, :512].double().numpy()
            for h in heads:
                e = C @ wd[h]
                bound = U_BF16 * np.abs(e) + 2.0 ** -14 * (np.abs(C) @ np.abs(wd[h]))
                err = np.abs(exp[which, b, :T, h] - e)
                assert (err <= bound).all(), (which, b, h, float(err.max()), float((err / bound).max()))
