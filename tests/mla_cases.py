"""Helpers shared by the GPU parity tests: put a seeded workload on the device, run the
CUDA path through the C ABI, and build the oracle's answer for chosen sequences."""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle as O
from mla_latent_kv_70_b300 import inputs as I

# Tolerances: bf16 inputs, fp32 accumulation.  Per output row (b,s,h):
# max_i |gpu - ref| / max_i |ref| <= 1e-2;  lse: |gpu - ref| <= 1e-3 absolute.
ROW_REL_TOL = 1e-2
LSE_ABS_TOL = 1e-3


class DeviceCase:
    """The tensors of one workload on the GPU (cache RoPE'd in place when the case asks)."""

    def __init__(self, case: I.DecodeCase, device="cuda"):
        import mla_latent_kv_70_b300 as mla
        self.case = case
        self.kv = I.cache(case, device=device)
        qn, qr = I.queries(case)
        self.q_nope, self.q_rope = qn.to(device), qr.to(device)
        w_uk, w_uv = I.weights(case)
        self.w_uk, self.w_uv = w_uk.to(device), w_uv.to(device)
        self.seqlens = torch.tensor(case.seqlens, dtype=torch.int32, device=device)
        self.block_table = case.block_table.to(device) if case.paged else None
        self.q_pos = case.q_positions().to(device) if case.rope else None
        if case.rope:
            # k^R carries RoPE at its own position (written once, at cache-append time);
            # a page pool's rows take the positions the block table gives them.
            if case.paged:
                pos = I.pool_positions(case).to(device)
            else:
                pos = torch.arange(case.t_cap, dtype=torch.int32, device=device).repeat(case.B)
            mla.mla_rope_inplace(self.kv, I.ROW, pos.numel(), I.D_C, pos, case.theta)

    def step(self, num_splits=None, max_seqlen=None, planned=False):
        """One DecodeStep; `planned` lets mla_decode_plan_splits pick the split count from
        the host-side lengths (as the bench does)."""
        import mla_latent_kv_70_b300 as mla
        c = self.case
        st = mla.DecodeStep(c.B, c.S, c.H, self.w_uk, self.w_uv,
                            max_seqlen=max_seqlen or max(c.seqlens),
                            num_splits=0 if planned else (c.num_splits if num_splits is None else num_splits),
                            causal=c.causal, rope_theta=c.theta, total_rows=c.total_tokens,
                            seqlens=c.seqlens if planned else None)
        st(self.q_nope, self.q_rope, self.kv, self.seqlens, block_table=self.block_table,
           q_pos=self.q_pos)
        torch.cuda.synchronize()
        return st


class DecodeOnlyCase:
    """The latent decode alone: seeded q_cat rows (inputs.q_cat) and the seeded cache on
    the GPU, with no absorption in front, so that the oracle and the kernel read the same
    bf16 query values and the comparison measures the decode's own arithmetic."""

    def __init__(self, case: I.DecodeCase, device="cuda"):
        assert not case.rope, "the decode reads rows as given; RoPE is checked on its own"
        self.case = case
        self.kv = I.cache(case, device=device)
        self.q_cat = I.q_cat(case).to(device)
        self.seqlens = torch.tensor(case.seqlens, dtype=torch.int32, device=device)
        self.block_table = case.block_table.to(device) if case.paged else None

    def run(self, num_splits=0, max_seqlen=None, noalloc=False):
        import mla_latent_kv_70_b300 as mla
        c = self.case
        max_seqlen = max_seqlen or max(c.seqlens)
        splits = num_splits or mla.mla_decode_num_splits(c.B, c.S, c.H, max_seqlen)
        o_lat = torch.full((c.B, c.S, c.H, I.D_C), float("nan"), device=self.kv.device)
        lse = torch.full((c.B, c.S, c.H), float("nan"), device=self.kv.device)
        status = torch.zeros(1, dtype=torch.int32, device=self.kv.device)
        kw = dict(scale=c.scale, max_seqlen=max_seqlen, block_table=self.block_table,
                  causal=c.causal, num_splits=splits, status=status)
        if noalloc:
            mla.mla_decode_latent_noalloc(self.q_cat, self.kv, self.seqlens, o_lat, lse, **kw)
        else:
            ws = mla.mla_decode_workspace_bytes(c.B, c.S, c.H, splits, max_seqlen)
            ws = torch.empty(ws // 4, device=self.kv.device) if ws else None
            mla.mla_decode_latent(self.q_cat, self.kv, self.seqlens, o_lat, lse, workspace=ws, **kw)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        return o_lat.cpu().numpy(), lse.cpu().numpy()


def oracle_decode_only(case: I.DecodeCase, b: int):
    """The oracle's absorbed attention (o_lat, lse) of sequence b on the seeded q_cat."""
    T = case.seqlens[b]
    rows = I.seq_rows(case, b)[:T].double().numpy()
    q = I.seq_q_cat(case, b).double().numpy()
    return O.decode_absorbed_seq(q[..., :I.D_C], q[..., I.D_C:], rows[:, :I.D_C],
                                 rows[:, I.D_C:], case.scale, case.causal)


def check_decode_only(case: I.DecodeCase, o_lat, lse, seqs, key=None):
    """o_lat rows within ROW_REL_TOL and every lse within LSE_ABS_TOL, whatever T."""
    for b in seqs:
        r_lat, r_lse = oracle_decode_only(case, b)
        assert row_rel_err(o_lat[b], r_lat) <= ROW_REL_TOL, (key, b)
        err = lse_err(lse[b], r_lse)
        log_lse(key, err, LSE_ABS_TOL)
        assert err <= LSE_ABS_TOL, (key, b, err)


def oracle_seq(case: I.DecodeCase, b: int, w_uk=None, w_uv=None, heads=None, expanded=False):
    """The oracle's (o_lat, lse, o) of sequence b, from the same seeded inputs."""
    T = case.seqlens[b]
    rows = I.seq_rows(case, b)[:T].double().numpy()
    C, KR = rows[:, :I.D_C], rows[:, I.D_C:]
    qn, qr = I.seq_queries(case, b)
    qn, qr = qn.double().numpy(), qr.double().numpy()
    if w_uk is None:
        w_uk, w_uv = (w.double().numpy() for w in I.weights(case))
    if heads is not None:
        qn, qr, w_uk, w_uv = qn[:, heads], qr[:, heads], w_uk[heads], w_uv[heads]
    if case.rope:
        KR = O.rope_interleaved(KR, np.arange(T), case.theta)
        pos = np.array([T - case.S + s for s in range(case.S)], dtype=np.float64)
        qr = O.rope_interleaved(qr, pos[:, None], case.theta)
    if expanded:
        o, lse = O.decode_expanded_seq(qn, qr, C, KR, w_uk, w_uv, case.scale, case.causal)
        return None, lse, o
    q_lat = O.absorb_q(qn, w_uk)
    o_lat, lse = O.decode_absorbed_seq(q_lat, qr, C, KR, case.scale, case.causal)
    return o_lat, lse, O.out_proj_uv(o_lat, w_uv)


# Query tokens that read at least SHORT_T rows (SHORT_T_ROPE when RoPE is applied) are
# held to LSE_ABS_TOL on the end-to-end path.  Below that, the bf16 rounding of q~ (and,
# with RoPE, of the rotated q^R and k^R), which the oracle does not make, reaches single
# scores that too few rows average out: lse_tolerance() bounds that part from the data.
# (The latent decode on its own is held to LSE_ABS_TOL at every length: see
# test_decode_only_gpu.py.)  The expected size of that part, for N(0,1) logits, is about
# 1.9e-4 (no RoPE) and 2.7e-4 (RoPE) standard deviation at 256 rows, shrinking as
# 1/sqrt(rows): the flat 1e-3 sits 5.3 standard deviations out at 256 rows without RoPE
# and 7.5 at 1024 rows with it.
SHORT_T = 256
SHORT_T_ROPE = 1024
U_BF16 = 2.0 ** -8                    # unit roundoff of bf16 (8 significant bits, RNE)
HOEFFDING_LAMBDA = 1e-6               # failure probability allowed per bounded quantity
K_HOEFFDING = math.sqrt(2.0 * math.log(2.0 / HOEFFDING_LAMBDA))

# Worst LSE error per test, |gpu - ref| and its ratio to the tolerance used; printed in
# the terminal summary (tests/conftest.py).
LSE_LOG: dict = {}


def current_test() -> str:
    """The running test's id (pytest sets PYTEST_CURRENT_TEST)."""
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


def log_lse(key, err: float, tol: float) -> None:
    key = key or current_test()
    old = LSE_LOG.get(key)
    ratio = err / tol if tol > 0 else 0.0
    if old is None or ratio > old[1]:
        LSE_LOG[key] = (err, ratio, tol)


def lse_tolerance(case: I.DecodeCase, b: int, w_uk=None) -> np.ndarray:
    """Per (s, h) bound on |lse_gpu - lse_exact| for the absorb -> decode path, [S, H].

    Rows of a query token that reads at least SHORT_T positions (SHORT_T_ROPE with RoPE)
    get LSE_ABS_TOL.  A token with fewer readable rows gets LSE_ABS_TOL (the decode's own
    arithmetic) plus the
    effect of roundings the oracle does not make: the CUDA path stores q~ = q_nope W_UK^T
    in bf16, and with RoPE also the rotated q^R and k^R.  Each such rounding moves a value
    v by e with |e| <= 2^-8 |v|; following the probabilistic model of rounding errors
    (independent, mean zero, bounded: Higham and Mary, "A new approach to probabilistic
    rounding error analysis", 2019), Hoeffding's inequality bounds a sum of n of them,
    sum_k c_k e_k, by sqrt(2 ln(2/lambda)) * sqrt(sum_k (c_k 2^-8 |v_k|)^2) with
    probability 1 - lambda.  To first order, lse moves by sum_j a_j d_j, d_j the change
    of the scaled score j and a the softmax weights; for q~ that is
    scale * sum_i e_i z_i with z = sum_j a_j c_j (the exact o_lat).  The second-order
    remainder is at most max_j d_j^2 / 2 (the Hessian of log-sum-exp is diag(a) - a a^T).
    """
    T = case.seqlens[b]
    S, H = case.S, case.H
    n_vis = [O.visible_length(T, S, s, case.causal) for s in range(S)]
    tol = np.full((S, H), LSE_ABS_TOL)
    limit = SHORT_T_ROPE if case.rope else SHORT_T
    short = [s for s in range(S) if 0 < n_vis[s] < limit]
    if not short:
        return tol
    rows = I.seq_rows(case, b)[:T].double().numpy()
    C, KR = rows[:, :I.D_C], rows[:, I.D_C:]
    qn, qr = (t.double().numpy() for t in I.seq_queries(case, b))
    if w_uk is None:
        w_uk = I.weights(case)[0].double().numpy()
    q_lat = O.absorb_q(qn, w_uk)
    if case.rope:
        KR = O.rope_interleaved(KR, np.arange(T), case.theta)
        pos = np.array([T - S + s for s in range(S)], dtype=np.float64)
        qr = O.rope_interleaved(qr, pos[:, None], case.theta)
    for s in short:
        n = n_vis[s]
        tol[s] = rounding_lse_tol(q_lat[s], qr[s], C[:n], KR[:n], case.scale, case.rope)
    return tol


def rounding_lse_tol(q_lat, q_rope, C, KR, scale, rope=False) -> np.ndarray:
    """LSE_ABS_TOL plus the bound of lse_tolerance for one query token (q_lat [H,512],
    q_rope [H,64]) over the rows C [n,512], KR [n,64] it reads: the q~ roundings (and,
    with RoPE, those of q^R and k^R) of the CUDA path, by Hoeffding's inequality, plus the
    second-order remainder.  Returns [H]."""
    u, k, sc = U_BF16, K_HOEFFDING, scale
    x = (q_lat @ C.T + q_rope @ KR.T) * sc                       # [H, n]
    a = np.exp(x - x.max(axis=1, keepdims=True))
    a /= a.sum(axis=1, keepdims=True)
    z = a @ C                                                    # [H, 512]
    var = ((u * q_lat * z) ** 2).sum(axis=1)                     # q~ roundings
    per_score = ((u * q_lat) ** 2) @ (C ** 2).T                  # [H, n]
    if rope:
        zr = a @ KR
        var += ((u * q_rope * zr) ** 2).sum(axis=1)              # q^R roundings
        var += (((a ** 2) @ (KR ** 2)) * (u * q_rope) ** 2).sum(axis=1)   # k^R roundings
        per_score += 2.0 * ((u * q_rope) ** 2) @ (KR ** 2).T
    first = k * sc * np.sqrt(var)
    second = 0.5 * (k * sc) ** 2 * per_score.max(axis=1)
    return LSE_ABS_TOL + first + second


def row_rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max|g - r| / max|r| along the last axis (rows with ref == 0 use abs)."""
    num = np.abs(gpu - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    den = np.where(den > 0, den, 1.0)
    return float((num / den).max()) if num.size else 0.0


def lse_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    both_inf = np.isneginf(gpu) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(gpu - ref))
    return float(d.max()) if d.size else 0.0


def check_lse(got: np.ndarray, ref: np.ndarray, tol, key=None, where=None) -> None:
    """|got - ref| <= tol elementwise (-inf matches -inf); logs the worst error and ratio."""
    with np.errstate(invalid="ignore"):
        d = np.where(np.isneginf(got) & np.isneginf(ref), 0.0, np.abs(got - ref))
    tol = np.broadcast_to(np.asarray(tol, dtype=np.float64), d.shape)
    if d.size:
        i = np.unravel_index(np.nanargmax(d / tol) if np.all(np.isfinite(d)) else 0, d.shape)
        log_lse(key, float(d[i]), float(tol[i]))
    assert np.all(d <= tol), (key or current_test(), where, float(np.nanmax(d)) if d.size else 0.0)


def check_case(dc: DeviceCase, st, seqs, expanded_heads=None):
    """o_lat and o of the sampled sequences within ROW_REL_TOL of the oracle; lse within
    lse_tolerance (LSE_ABS_TOL for every query token reading >= 256 rows)."""
    case = dc.case
    w_uk, w_uv = (w.double().numpy() for w in I.weights(case))
    o_lat = st.o_lat.cpu().numpy()
    lse = st.lse.cpu().numpy()
    o = st.o.cpu().numpy()
    assert int(st.status.item()) == 0
    for b in seqs:
        r_lat, r_lse, r_o = oracle_seq(case, b, w_uk, w_uv)
        tol = lse_tolerance(case, b, w_uk)
        assert row_rel_err(o_lat[b], r_lat) <= ROW_REL_TOL, (case.name, b)
        check_lse(lse[b], r_lse, tol, where=(case.name, b))
        assert row_rel_err(o[b], r_o) <= ROW_REL_TOL, (case.name, b)
        if expanded_heads is not None and b == list(seqs)[0]:
            _, e_lse, e_o = oracle_seq(case, b, w_uk, w_uv, heads=expanded_heads, expanded=True)
            assert row_rel_err(o[b][:, expanded_heads], e_o) <= ROW_REL_TOL
            check_lse(lse[b][:, expanded_heads], e_lse, tol[:, expanded_heads],
                      where=(case.name, "expanded", b))
