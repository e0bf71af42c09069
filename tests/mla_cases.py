"""Helpers shared by the GPU parity tests: put a seeded workload on the device, run the
CUDA path through the C ABI, and build the oracle's answer for chosen sequences."""
from __future__ import annotations

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
            # k^R carries RoPE at its own position (written once, at cache-append time).
            assert not case.paged
            rows = case.B * case.t_cap
            pos = torch.arange(case.t_cap, dtype=torch.int32, device=device).repeat(case.B)
            mla.mla_rope_inplace(self.kv, I.ROW, rows, I.D_C, pos, case.theta)

    def step(self, num_splits=None, max_seqlen=None):
        import mla_latent_kv_70_b300 as mla
        c = self.case
        st = mla.DecodeStep(c.B, c.S, c.H, self.w_uk, self.w_uv,
                            max_seqlen=max_seqlen or max(c.seqlens),
                            num_splits=c.num_splits if num_splits is None else num_splits,
                            causal=c.causal, rope_theta=c.theta, total_rows=c.total_tokens)
        st(self.q_nope, self.q_rope, self.kv, self.seqlens, block_table=self.block_table,
           q_pos=self.q_pos)
        torch.cuda.synchronize()
        return st


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


def lse_rounding_bound(case: I.DecodeCase, b: int, w_uk=None) -> np.ndarray:
    """Bound on |lse_gpu - lse_exact| from the bf16 roundings of the CUDA path, per (s, h).

    bf16 keeps 8 significant bits, so one rounding moves a value by at most 2^-8 of
    its magnitude.  The CUDA path rounds q~ = q_nope W_UK^T to bf16 before scoring, and
    the half of each score computed by the peer CTA travels as bf16: together these move
    the score of row j by at most 2 * 2^-8 * sum_i |q~_i c_ji|.  With RoPE, q^R and k^R
    are each rotated and stored as bf16 (two more roundings of the rope term).
    Log-sum-exp moves by at most the largest scaled score change.  The bound below
    doubles that to cover the fp32 accumulations and the exp2 approximation.  At small T
    it exceeds 1e-3; for the named workloads (T >= 256) the tests use 1e-3.
    """
    T = case.seqlens[b]
    if T == 0:
        return np.zeros((case.S, case.H))
    rows = I.seq_rows(case, b)[:T].double().numpy()
    qn, qr = I.seq_queries(case, b)
    if w_uk is None:
        w_uk = I.weights(case)[0].double().numpy()
    q_lat = np.abs(O.absorb_q(qn.double().numpy(), w_uk))       # [S,H,512]
    terms = q_lat @ np.abs(rows[:, :I.D_C]).T                    # [S,H,T]
    if case.rope:
        # q^R and k^R are both rotated and stored as bf16 on the GPU: 2 more roundings.
        terms = terms + 2.0 * np.abs(qr.double().numpy()) @ np.abs(rows[:, I.D_C:]).T
    return case.scale * 2.0 * (2.0 * 2.0 ** -8) * terms.max(axis=-1)


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
