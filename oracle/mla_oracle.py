"""Plain fp64 CPU oracle for Multi-Head Latent Attention decode with weight absorption.

TEST INFRASTRUCTURE ONLY.  This module is imported by the test suite, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``.  The
product path (the ``mla_latent_kv_70_b300`` package and its CUDA library) never
imports, links or calls it, and it imports nothing from the product.

Everything is float64 numpy.  Inputs arrive as float arrays whose values are the
exact bf16 inputs of the GPU path (bf16 -> float64 is exact); nothing here rounds
to a narrower type.  Dimensions are read from the array shapes, so the same code
runs the pages' toy examples (d_c=3, d_k=d_r=2) and the DeepSeek-V3 shapes
(d_c=512, d_r=64, d_nope=d_v=128).

Pages cited (by title):
  [MLA]     "Multi-Head Latent Attention (MLA)" (molayo1419.me)
  [CALC]    "MLA의 계산: KV를 펼치지 않고 Attention하기" (ai-systems-engineering.com)
  [ANATOMY] "DeepSeek Multi-Head Latent Attention(MLA) 아키텍처 해부" (blog.huny.dev)

Readings taken where the pages are silent or disagree (each is also listed in the
design notes): one score scale 1/sqrt(d_nope + d_r) ([CALC], "RoPE 경로를 분리한
이유"); one decoupled RoPE key k^R shared by all heads, cached beside c^KV
([CALC], Fig. 2; [ANATOMY] section 2); W_UK[h] and W_UV[h] stored as
[d_c x d_k] matrices with K_h = C W_UK[h] ([MLA], "공식 정의"); RoPE on
interleaved pairs with inverse frequency theta^(-2i/d_r) ([MLA], "구현",
_apply_rope); natural-log LSE; an empty sequence gives o = 0 and lse = -inf.

Parity pins for every function live in tests/test_oracle_pins.py; none of them is
"parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "score_scale",
    "rope_interleaved",
    "absorb_q",
    "visible_length",
    "decode_expanded_seq",
    "decode_absorbed_seq",
    "decode_absorbed_partial_seq",
    "combine_partials",
    "out_proj_uv",
    "gather_paged_rows",
    "append_latent_rows",
    "fuse_query_weights",
    "fuse_output_weights",
    "absorb_q_from_latent",
    "out_proj_fused",
    "out_proj_heads",
    "e4m3_decode",
    "e4m3_encode",
    "fp8_row_scale",
    "quantize_fp8_rows",
    "dequantize_fp8_rows",
    "cache_values_per_token",
    "cache_bytes_per_token",
    "compression_ratio",
    "full_cache_gib",
]


# ----------------------------------------------------------------------------
# Scale and positions
# ----------------------------------------------------------------------------

def score_scale(d_nope: int, d_r: int) -> float:
    """1 / sqrt(d_content + d_rope).

    [CALC] "Content 점수와 위치 점수 합치기": the toy query/key have a 2-wide content
    part and a 2-wide position part, so the scores are divided by sqrt(2+2) = 2.
    [CALC] "RoPE 경로를 분리한 이유": after absorption the content dot runs in the
    d_c-wide latent space, but the scale stays sqrt(d_content + d_rope), not
    sqrt(d_c + d_rope), because the score itself is unchanged.
    """
    return 1.0 / math.sqrt(d_nope + d_r)


def visible_length(T: int, S: int, s: int, causal: bool) -> int:
    """Number of cached positions query token s (of S) may read.

    The sequence holds T cached rows at positions 0..T-1 and the S query tokens
    are its last S rows ([CALC] "계산 재배치의 효과와 한계": the current token's latent
    is appended before attention and the token reads itself).  Without a mask
    every query reads all T rows; with the causal mask of [CALC] "Content 점수와
    위치 점수 합치기" (several tokens computed together must not read future
    positions) query s sits at position T-S+s and reads rows 0..T-S+s.
    """
    if T <= 0:
        return 0
    if not causal:
        return T
    return max(0, min(T, T - S + s + 1))


def rope_interleaved(x: np.ndarray, pos, theta: float = 10000.0) -> np.ndarray:
    """Rotate interleaved pairs (x[2i], x[2i+1]) by angle pos * theta^(-2i/d).

    [MLA] "구현" (_apply_rope): the inverse frequencies are theta^(-(0,2,4,..)/d_r),
    the angle is position x inverse frequency, and the even/odd elements of the
    last axis form the rotated pairs (x1 cos - x2 sin, x1 sin + x2 cos).
    ``pos`` broadcasts against x[..., 0].
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    if d % 2:
        raise ValueError("rope width must be even")
    inv_freq = np.power(float(theta), -np.arange(0, d, 2, dtype=np.float64) / d)
    angle = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    cos, sin = np.cos(angle), np.sin(angle)
    even, odd = x[..., 0::2], x[..., 1::2]
    out = np.empty(np.broadcast_shapes(x.shape, angle.shape[:-1] + (d,)), dtype=np.float64)
    out[..., 0::2] = even * cos - odd * sin
    out[..., 1::2] = even * sin + odd * cos
    return out


# ----------------------------------------------------------------------------
# Key absorption (step a1)
# ----------------------------------------------------------------------------

def absorb_q(q_nope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """q_lat[..., h, :] = q_nope[..., h, :] . W_UK[h]^T.

    [CALC] "Key 투영을 Query 쪽으로 옮기기" (Fig. 3): q (c_j U^K)^T = (q U^K^T) c_j^T,
    so the per-head content query is mapped once into the latent space
    (q~ = q U^K^T, 1 x d_c) instead of expanding every cached latent.
    q_nope: [..., H, d_nope]; w_uk: [H, d_c, d_nope]  ->  [..., H, d_c].
    """
    q = np.asarray(q_nope, dtype=np.float64)
    w = np.asarray(w_uk, dtype=np.float64)
    return np.einsum("...hk,hck->...hc", q, w)


# ----------------------------------------------------------------------------
# The definition: textbook attention over expanded per-head K/V
# ----------------------------------------------------------------------------

def decode_expanded_seq(q_nope, q_rope, c_kv, k_rope, w_uk, w_uv, scale, causal=False):
    """One sequence, expanded form (the definition the absorbed method must equal).

    [MLA] "공식 정의": K_h = c^KV W_UK^(h), V_h = c^KV W_UV^(h).
    [CALC] "Content 점수와 위치 점수 합치기" (Fig. 2): s_j = q^C_h . k^C_{j,h} + q^R_h . k^R_j
    (no cross terms; k^R is shared by the heads), divided by the scale, softmax
    over all readable positions (one softmax over the positions, not one per
    position), then the attention weights mix the per-head values v_{j,h}; the
    position key is never appended to the value.

    q_nope [S,H,d_nope]; q_rope [S,H,d_r] (already rotated); c_kv [T,d_c];
    k_rope [T,d_r] (already rotated); w_uk, w_uv [H,d_c,d_k].
    Returns o [S,H,d_v] and lse [S,H] (natural log of sum_j exp(scale*s_j)).
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    C = np.asarray(c_kv, np.float64)
    KR = np.asarray(k_rope, np.float64)
    w_uk = np.asarray(w_uk, np.float64)
    w_uv = np.asarray(w_uv, np.float64)
    S, H, _ = q_nope.shape
    T = C.shape[0]
    d_v = w_uv.shape[2]
    o = np.zeros((S, H, d_v))
    lse = np.full((S, H), -np.inf)
    for h in range(H):
        K_h = C @ w_uk[h]          # [T, d_k] content keys of head h
        V_h = C @ w_uv[h]          # [T, d_v] values of head h
        for s in range(S):
            n = visible_length(T, S, s, causal)
            if n == 0:
                continue
            x = (K_h[:n] @ q_nope[s, h] + KR[:n] @ q_rope[s, h]) * scale
            m = x.max()
            e = np.exp(x - m)
            l = e.sum()
            a = e / l
            o[s, h] = a @ V_h[:n]
            lse[s, h] = m + math.log(l)
    return o, lse


# ----------------------------------------------------------------------------
# The absorbed form (steps a2-a4): scores and aggregation in latent space
# ----------------------------------------------------------------------------

def decode_absorbed_partial_seq(q_lat, q_rope, c_kv, k_rope, scale, t0, t1, n_visible):
    """Attention of every (s, h) over cached rows [t0, min(t1, n_visible[s])).

    [CALC] "Key 투영을 Query 쪽으로 옮기기": content score = q~ . c_j read straight
    from the latent cache; plus the position score q^R . k^R_j ("RoPE 경로를
    분리한 이유": the position part is computed separately and added).
    [CALC] "Value 투영을 가중합 뒤로 옮기기" (Fig. 4): z = a C, the latents mixed
    with the attention weights, is returned as o_lat (U^V is applied later).

    Returns (o_lat [S,H,d_c] normalised over the rows it saw, lse [S,H]); rows it
    never saw give o_lat = 0, lse = -inf.
    """
    q_lat = np.asarray(q_lat, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    C = np.asarray(c_kv, np.float64)
    KR = np.asarray(k_rope, np.float64)
    S, H, d_c = q_lat.shape
    o_lat = np.zeros((S, H, d_c))
    lse = np.full((S, H), -np.inf)
    for s in range(S):
        hi = min(t1, n_visible[s])
        if hi <= t0:
            continue
        Cs, KRs = C[t0:hi], KR[t0:hi]
        x = (q_lat[s] @ Cs.T + q_rope[s] @ KRs.T) * scale    # [H, n]
        m = x.max(axis=1, keepdims=True)
        e = np.exp(x - m)
        l = e.sum(axis=1, keepdims=True)
        o_lat[s] = (e / l) @ Cs
        lse[s] = (m + np.log(l))[:, 0]
    return o_lat, lse


def decode_absorbed_seq(q_lat, q_rope, c_kv, k_rope, scale, causal=False):
    """One sequence, absorbed form over all readable rows: (o_lat [S,H,d_c], lse [S,H])."""
    q_lat = np.asarray(q_lat, np.float64)
    S = q_lat.shape[0]
    T = np.asarray(c_kv).shape[0]
    n_vis = [visible_length(T, S, s, causal) for s in range(S)]
    return decode_absorbed_partial_seq(q_lat, q_rope, c_kv, k_rope, scale, 0, T, n_vis)


def combine_partials(o_parts, lse_parts):
    """Merge attention over disjoint row ranges by their log-sum-exp.

    Not on the pages (split-KV serves long contexts at small batch).  It follows
    from the softmax definition: if part k has lse_k and normalised output o_k,
    the whole has lse = log sum_k exp(lse_k) and o = sum_k exp(lse_k - lse) o_k.
    o_parts [K,...,d]; lse_parts [K,...].  All parts empty -> o = 0, lse = -inf.
    """
    o_parts = np.asarray(o_parts, np.float64)
    lse_parts = np.asarray(lse_parts, np.float64)
    m = lse_parts.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - m_safe), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), -np.inf)
    coef = np.where(finite, 1.0 / np.where(finite, tot, 1.0), 0.0)
    o = np.einsum("k...,k...d->...d", w * coef, o_parts)
    return o, lse


# ----------------------------------------------------------------------------
# Value up-projection (step a6)
# ----------------------------------------------------------------------------

def out_proj_uv(o_lat: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """o[..., h, :] = o_lat[..., h, :] . W_UV[h].

    [CALC] "Value 투영을 가중합 뒤로 옮기기": a (C U^V) = (a C) U^V = z U^V, so U^V is
    applied once, per head, after the latents are mixed.
    o_lat [..., H, d_c]; w_uv [H, d_c, d_v] -> [..., H, d_v].
    """
    return np.einsum("...hc,hcv->...hv", np.asarray(o_lat, np.float64),
                     np.asarray(w_uv, np.float64))


# ----------------------------------------------------------------------------
# Pre-fused weights ([CALC] "Query·출력 투영과 합치기")
# ----------------------------------------------------------------------------

def fuse_query_weights(w_uq, w_uk):
    """W_UQK[h] = W_UQ[h] W_UK[h]^T, the query projection and the transposed key
    projection multiplied ahead of time ([CALC] "Query·출력 투영과 합치기": U^Q is 3x2 and
    (U^K)^T 2x3 in the toy, so their product is a 3x3 matrix that takes c^Q straight to
    q~).  w_uq [H, d_cq, d_k]; w_uk [H, d_c, d_k] -> [H, d_cq, d_c]."""
    return np.einsum("hik,hck->hic", np.asarray(w_uq, np.float64), np.asarray(w_uk, np.float64))


def fuse_output_weights(w_uv, w_o):
    """W_UVO[h] = W_UV[h] W_O[h], the value projection multiplied into head h's rows of
    the output projection ([CALC] "Query·출력 투영과 합치기": U^V 3x2 times W^O_1 2x8 gives
    the 3x8 matrix that takes z to head 1's contribution to the model dimension).
    w_uv [H, d_c, d_v]; w_o [H, d_v, d_model] -> [H, d_c, d_model]."""
    return np.einsum("hcv,hvj->hcj", np.asarray(w_uv, np.float64), np.asarray(w_o, np.float64))


def absorb_q_from_latent(c_q, w_uqk):
    """q~[..., h, :] = c^Q[..., :] W_UQK[h]: the content query of every head taken from the
    query latent in one product.  c_q [..., d_cq]; w_uqk [H, d_cq, d_c] -> [..., H, d_c]."""
    return np.einsum("...i,hic->...hc", np.asarray(c_q, np.float64), np.asarray(w_uqk, np.float64))


def out_proj_fused(o_lat, w_uvo):
    """out[..., :] = sum_h z_h W_UVO[h]: every head's contribution to the model dimension,
    summed ([CALC] "Query·출력 투영과 합치기": the heads' contributions add up to the whole
    output projection).  o_lat [..., H, d_c]; w_uvo [H, d_c, d_model] -> [..., d_model]."""
    return np.einsum("...hc,hcj->...j", np.asarray(o_lat, np.float64), np.asarray(w_uvo, np.float64))


def out_proj_heads(o, w_o):
    """The output projection of per-head outputs: out = sum_h o_h W_O[h] (the unfused
    order).  o [..., H, d_v]; w_o [H, d_v, d_model] -> [..., d_model]."""
    return np.einsum("...hv,hvj->...j", np.asarray(o, np.float64), np.asarray(w_o, np.float64))


# ----------------------------------------------------------------------------
# Paged cache addressing
# ----------------------------------------------------------------------------

def gather_paged_rows(pool: np.ndarray, block_row: np.ndarray, T: int) -> np.ndarray:
    """Rows 0..T-1 of one sequence stored in pages of a shared pool.

    [MLA] "MLA + 투기적 디코딩", "vLLM 구현 과제": paged serving of MLA needs a page
    table whose entries hold latent vectors instead of K/V pairs.  Row t lives in page block_row[t // P] at
    offset t % P, with P = pool.shape[1].
    """
    pool = np.asarray(pool)
    P = pool.shape[1]
    t = np.arange(T)
    return pool[np.asarray(block_row)[t // P], t % P]


def append_latent_rows(new_rows, start: int, theta=None, d_r: int = 64):
    """The cache rows one sequence gains in a decode step, and their positions.

    [CALC] "계산 재배치의 효과와 한계": the current token's latent is added to the cache
    before attention, so the S new rows take positions start .. start + S - 1 (start = the
    rows already cached) and each query token then reads itself.  [ANATOMY] section 2:
    the cached k^R carries RoPE, so the k^R part of the row at position t is rotated by t
    when the row is written (theta None or 0: stored as given); c^KV is stored unchanged.
    new_rows [S, d_c + d_r] (the last d_r values are k^R).
    Returns (rows [S, d_c + d_r] as stored, positions [S]).
    """
    rows = np.array(new_rows, dtype=np.float64)
    pos = start + np.arange(rows.shape[0])
    if theta:
        rows[:, -d_r:] = rope_interleaved(rows[:, -d_r:], pos, theta)
    return rows, pos


# ----------------------------------------------------------------------------
# Cache-size identities
# ----------------------------------------------------------------------------

# ----------------------------------------------------------------------------
# FP8 latent cache ([ANATOMY] section 5, the checklist item on FP8 mixed precision:
# E4M3 applied to the 512-wide latent space with a per-token or per-tensor scale).
# The pages fix neither the E4M3 encoding nor the scale rule; the readings here:
#   * E4M3 is the OCP 8-bit floating point format "E4M3": sign, 4 exponent bits with
#     bias 7, 3 mantissa bits, subnormals at exponent field 0 (value m/8 * 2^-6), no
#     infinities, S.1111.111 the only NaN, largest finite 448;
#   * one scale per cached token over its 512 latent values, a power of two: the
#     smallest 2^e with amax/2^e <= 448 (e clamped to [-126, 15]; an all-zero row
#     takes 2^0), so that dividing by it and multiplying back are exact, and 2^112 * 2^e
#     stays a finite bf16 (the factor the GPU path widens E4M3 values to bf16 with);
#     a row whose amax exceeds 448 * 2^15 saturates;
#   * codes are the round-to-nearest-even E4M3 value of c/scale, saturating at +-448;
#   * the 64-wide RoPE key k^R stays as it is (bf16): the checklist speaks of the
#     latent space only.
# ----------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Values of E4M3 codes (uint8) as float64; NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


_E4M3_POS = e4m3_decode(np.arange(0x7F))          # the 127 finite non-negative values, increasing


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even E4M3 codes of finite float64 values, saturating at +-448.

    Nearest by brute force over the 127 non-negative values; a tie goes to the code
    with an even mantissa (its lowest bit 0).  The sign bit is the sign of x (so a
    negative value that rounds to zero gives 0x80)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x).reshape(-1)
    d = np.abs(a[:, None] - _E4M3_POS[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    n_cand = cand.sum(axis=1)
    first = cand.argmax(axis=1)
    last = _E4M3_POS.size - 1 - cand[:, ::-1].argmax(axis=1)
    code = np.where((n_cand > 1) & (first % 2 == 1), last, first)   # ties: the even code
    code = np.where(a >= 448.0, 0x7E, code)
    code = code | np.where(np.signbit(x.reshape(-1)), 0x80, 0)
    return code.astype(np.uint8).reshape(x.shape)


def fp8_row_scale(c_row) -> float:
    """Per-token scale: the smallest power of two 2^e with max|c|/2^e <= 448."""
    amax = float(np.max(np.abs(np.asarray(c_row, dtype=np.float64))))
    if amax == 0.0:
        return 1.0
    mant, e = math.frexp(amax / 448.0)          # amax/448 = mant * 2^e, 0.5 <= mant < 1
    if mant == 0.5:                             # an exact power of two
        e -= 1
    return math.ldexp(1.0, min(15, max(-126, e)))


def quantize_fp8_rows(rows, d_c: int = 512):
    """Cache rows [n, d_c + d_r] -> (codes uint8 [n, d_c], k^R [n, d_r] unchanged,
    scales [n]): codes = E4M3(c / scale) per row."""
    rows = np.asarray(rows, dtype=np.float64)
    scales = np.array([fp8_row_scale(r[:d_c]) for r in rows], dtype=np.float64)
    codes = e4m3_encode(rows[:, :d_c] / scales[:, None])
    return codes, rows[:, d_c:].copy(), scales


def dequantize_fp8_rows(codes, k_rope, scales) -> np.ndarray:
    """Cache rows [n, d_c + d_r] read back from the FP8 form: scale * E4M3 value, then k^R."""
    c = e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, None]
    return np.concatenate([c, np.asarray(k_rope, dtype=np.float64)], axis=1)


def cache_values_per_token(kind: str, n_h=128, d_k=128, d_c=512, d_r=64, n_kv_heads=8) -> int:
    """Cached values per token per layer.

    [MLA] "공식 정의": MHA caches 2 n_h d_k values per token.
    [ANATOMY] section 1 table: GQA caches K and V for its KV heads only; MLA caches
    the 512-wide c^KV plus the 64-wide shared k^R (576 values).
    """
    if kind == "mha":
        return 2 * n_h * d_k
    if kind == "gqa":
        return 2 * n_kv_heads * d_k
    if kind == "mla":
        return d_c + d_r
    raise ValueError(kind)


def cache_bytes_per_token(kind: str, bytes_per_value: int = 2, **dims) -> int:
    """FP16/bf16 bytes cached per token per layer ([ANATOMY] section 1 table)."""
    return cache_values_per_token(kind, **dims) * bytes_per_value


def compression_ratio(n_h=128, d_k=128, d_c=512) -> float:
    """2 n_h d_k / d_c ([MLA] "공식 정의", compression ratio)."""
    return 2 * n_h * d_k / d_c


def full_cache_gib(kind: str, tokens: int = 131072, layers: int = 61, **dims) -> float:
    """Whole-model cache size in GiB ([ANATOMY] section 1 table, 128k context, 61 layers)."""
    return cache_bytes_per_token(kind, **dims) * tokens * layers / 2.0 ** 30
