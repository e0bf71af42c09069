"""Pins for the fp64 oracle: the pages' worked numbers, closed forms, invariants, brute force.

Each test ties the oracle to something other than itself: a value printed on the
pages (fixtures under tests/golden/, each with its citation), a closed form, an
invariant of softmax/RoPE, or an explicit pure-Python loop on a tiny case.
The last group plants mistakes into copies of the oracle's steps and checks that
the pins notice them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def toy_single_row(g):
    """The worked example as a 1-head, 1-query, 1-row problem (d_c=3, d_nope=d_r=2)."""
    q_nope = np.array(g["q_content"], float).reshape(1, 1, 2)
    q_rope = np.array(g["q_rope"], float).reshape(1, 1, 2)
    c = np.array([g["latent_c"]], float)
    kr = np.array([g["k_rope"]], float)
    w_uk = np.array(g["w_uk_selects_first_two"], float)[None]
    return q_nope, q_rope, c, kr, w_uk


# ----------------------------------------------------------------------------
# Values printed on the pages
# ----------------------------------------------------------------------------

def test_toy_score_scale_and_sum():
    g = gold("toy_score.json")
    assert O.score_scale(2, 2) == pytest.approx(1.0 / g["scale_divisor"], abs=0)
    # the latent width (3) must not enter the scale
    assert O.score_scale(2, 2) != pytest.approx(1.0 / math.sqrt(3 + 2))
    q_nope, q_rope, c, kr, w_uk = toy_single_row(g)
    scale = O.score_scale(2, 2)
    w_uv = np.eye(3)[:, :2][None]
    # With one readable row the log-sum-exp is that row's scaled score.
    _, lse_e = O.decode_expanded_seq(q_nope, q_rope, c, kr, w_uk, w_uv, scale)
    q_lat = O.absorb_q(q_nope, w_uk)
    _, lse_a = O.decode_absorbed_seq(q_lat, q_rope, c, kr, scale)
    assert lse_e[0, 0] == pytest.approx(g["scaled_score"], abs=1e-15)
    assert lse_a[0, 0] == pytest.approx(g["scaled_score"], abs=1e-15)
    # Add a second row with zero latent and zero rope key: score 0.
    c2 = np.vstack([c, np.zeros(3)])
    kr2 = np.vstack([kr, np.zeros(2)])
    _, lse2 = O.decode_absorbed_seq(q_lat, q_rope, c2, kr2, scale)
    assert lse2[0, 0] == pytest.approx(math.log(math.exp(g["scaled_score"]) + 1.0), abs=1e-15)


def test_toy_score_parts():
    g = gold("toy_score.json")
    q_nope, q_rope, c, kr, w_uk = toy_single_row(g)
    content_key = c @ w_uk[0]
    assert float(content_key[0] @ q_nope[0, 0]) == g["content_score"]
    assert float(kr[0] @ q_rope[0, 0]) == pytest.approx(g["rope_score"], abs=1e-15)
    # scale 1: the oracle's raw score is the plain sum, no cross terms
    _, lse = O.decode_absorbed_seq(O.absorb_q(q_nope, w_uk), q_rope, c, kr, 1.0)
    assert lse[0, 0] == pytest.approx(g["score"], abs=1e-14)


def test_toy_key_absorption():
    g = gold("toy_key_absorption.json")
    w_uk = np.array(g["w_uk_selects_first_two"], float)[None]
    q = np.array(g["q"], float).reshape(1, 2)
    c3 = np.array(g["latent_c3"], float)
    q_tilde = O.absorb_q(q, w_uk)[0]
    assert q_tilde.tolist() == g["q_tilde"]
    assert float(q_tilde @ c3) == g["score"]
    assert (c3 @ w_uk[0]).tolist() == g["content_key"]
    assert float((c3 @ w_uk[0]) @ q[0]) == g["score"]


def test_toy_value_absorption():
    g = gold("toy_value_absorption.json")
    C = np.array(g["latents"], float)
    w = np.array(g["weights"], float)
    w_uv = np.array(g["w_uv"], float)[None]
    assert (C @ w_uv[0]).tolist() == g["values"]
    # Impose the table's weights through the position score: content query 0,
    # rope query [1,0], rope keys [ln(w_j)/scale, 0]  =>  softmax = w (sum w = 1).
    scale = O.score_scale(2, 2)
    q_nope = np.zeros((1, 1, 2))
    q_rope = np.array([1.0, 0.0]).reshape(1, 1, 2)
    kr = np.stack([np.log(w) / scale, np.zeros(4)], axis=1)
    w_uk = np.zeros((1, 3, 2))
    o, _ = O.decode_expanded_seq(q_nope, q_rope, C, kr, w_uk, w_uv, scale)
    np.testing.assert_allclose(o[0, 0], g["output"], rtol=0, atol=1e-14)
    o_lat, lse = O.decode_absorbed_seq(O.absorb_q(q_nope, w_uk), q_rope, C, kr, scale)
    np.testing.assert_allclose(o_lat[0, 0], g["z"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(O.out_proj_uv(o_lat, w_uv)[0, 0], g["output"], rtol=0, atol=1e-14)
    assert lse[0, 0] == pytest.approx(0.0, abs=1e-14)   # log(sum w) = 0


def test_cache_identities():
    g = gold("cache_identities.json")
    d = dict(n_h=g["n_h"], d_k=g["d_k"], d_c=g["d_c"], d_r=g["d_r"], n_kv_heads=g["gqa_kv_heads"])
    assert O.compression_ratio(g["n_h"], g["d_k"], g["d_c"]) == g["compression_ratio"]
    assert O.cache_values_per_token("mla", **d) == g["mla_values_per_token"]
    for kind, nbytes in g["bytes_per_token_fp16"].items():
        assert O.cache_bytes_per_token(kind, **d) == nbytes
    mla = O.cache_bytes_per_token("mla", **d)
    assert 100 * (1 - mla / O.cache_bytes_per_token("mha", **d)) == pytest.approx(
        g["savings_percent"]["vs_mha"], abs=0.005)
    assert 100 * (1 - mla / O.cache_bytes_per_token("gqa", **d)) == pytest.approx(
        g["savings_percent"]["vs_gqa"], abs=0.006)
    for kind, gb in g["full_cache_gb"].items():
        assert O.full_cache_gib(kind, g["context_tokens"], g["layers"], **d) == pytest.approx(gb, abs=0.005)


# ----------------------------------------------------------------------------
# Brute force: explicit loops on tiny inputs
# ----------------------------------------------------------------------------

def brute_force(q_nope, q_rope, C, KR, w_uk, w_uv, scale, causal):
    """Textbook attention written as scalar loops, no numpy linear algebra."""
    S, H, dk = len(q_nope), len(q_nope[0]), len(q_nope[0][0])
    T = len(C)
    dc = len(C[0]) if T else len(w_uk[0])
    dr = len(q_rope[0][0])
    dv = len(w_uv[0][0])
    o = [[[0.0] * dv for _ in range(H)] for _ in range(S)]
    lse = [[-math.inf] * H for _ in range(S)]
    for s in range(S):
        n = T if not causal else T - S + s + 1
        for h in range(H):
            xs = []
            for j in range(n):
                sc = 0.0
                for k in range(dk):
                    key = sum(C[j][i] * w_uk[h][i][k] for i in range(dc))
                    sc += q_nope[s][h][k] * key
                for r in range(dr):
                    sc += q_rope[s][h][r] * KR[j][r]
                xs.append(sc * scale)
            if not xs:
                continue
            m = max(xs)
            den = sum(math.exp(x - m) for x in xs)
            for v in range(dv):
                acc = 0.0
                for j in range(n):
                    val = sum(C[j][i] * w_uv[h][i][v] for i in range(dc))
                    acc += math.exp(xs[j] - m) / den * val
                o[s][h][v] = acc
            lse[s][h] = m + math.log(den)
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("causal,S,T", [(False, 1, 5), (True, 2, 6), (True, 3, 3), (False, 2, 1)])
def test_brute_force_tiny(causal, S, T):
    rng = np.random.default_rng(7 + S * 10 + T)
    H, dc, dk, dr, dv = 2, 4, 3, 2, 3
    q_nope = rng.standard_normal((S, H, dk))
    q_rope = rng.standard_normal((S, H, dr))
    C = rng.standard_normal((T, dc))
    KR = rng.standard_normal((T, dr))
    w_uk = rng.standard_normal((H, dc, dk))
    w_uv = rng.standard_normal((H, dc, dv))
    scale = O.score_scale(dk, dr)
    o_ref, lse_ref = brute_force(q_nope.tolist(), q_rope.tolist(), C.tolist(), KR.tolist(),
                                 w_uk.tolist(), w_uv.tolist(), scale, causal)
    o_e, lse_e = O.decode_expanded_seq(q_nope, q_rope, C, KR, w_uk, w_uv, scale, causal)
    np.testing.assert_allclose(o_e, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse_e, lse_ref, rtol=1e-12, atol=1e-13)
    o_lat, lse_a = O.decode_absorbed_seq(O.absorb_q(q_nope, w_uk), q_rope, C, KR, scale, causal)
    np.testing.assert_allclose(O.out_proj_uv(o_lat, w_uv), o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse_a, lse_ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------
# Absorbed == expanded (the pages claim equality to ~1e-14)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("S,H,T,causal", [(1, 4, 300, False), (2, 3, 129, True), (1, 16, 64, False)])
def test_absorbed_equals_expanded_ds_dims(S, H, T, causal):
    rng = np.random.default_rng(S * 1000 + H * 10 + T)
    q_nope = rng.standard_normal((S, H, 128))
    q_rope = rng.standard_normal((S, H, 64))
    C = rng.standard_normal((T, 512))
    KR = rng.standard_normal((T, 64))
    w_uk = rng.standard_normal((H, 512, 128)) / math.sqrt(512)
    w_uv = rng.standard_normal((H, 512, 128)) / math.sqrt(512)
    scale = O.score_scale(128, 64)
    o_e, lse_e = O.decode_expanded_seq(q_nope, q_rope, C, KR, w_uk, w_uv, scale, causal)
    o_lat, lse_a = O.decode_absorbed_seq(O.absorb_q(q_nope, w_uk), q_rope, C, KR, scale, causal)
    o_a = O.out_proj_uv(o_lat, w_uv)
    rel = np.abs(o_a - o_e).max() / np.abs(o_e).max()
    assert rel < 1e-12
    assert np.abs(lse_a - lse_e).max() < 1e-12


# ----------------------------------------------------------------------------
# Closed forms and invariants of the softmax
# ----------------------------------------------------------------------------

def rand_seq(rng, S, H, T, dc=16, dr=4):
    return (rng.standard_normal((S, H, dc)), rng.standard_normal((S, H, dr)),
            rng.standard_normal((T, dc)), rng.standard_normal((T, dr)))


def test_single_row_closed_form():
    rng = np.random.default_rng(1)
    q_lat, q_rope, C, KR = rand_seq(rng, 1, 3, 1)
    o_lat, lse = O.decode_absorbed_seq(q_lat, q_rope, C, KR, 0.25)
    for h in range(3):
        np.testing.assert_array_equal(o_lat[0, h], C[0])
        assert lse[0, h] == pytest.approx(0.25 * (q_lat[0, h] @ C[0] + q_rope[0, h] @ KR[0]), abs=1e-14)


def test_identical_rows_uniform_weights():
    rng = np.random.default_rng(2)
    q_lat, q_rope, C, KR = rand_seq(rng, 1, 2, 1)
    T = 37
    o_lat, lse = O.decode_absorbed_seq(q_lat, q_rope, np.repeat(C, T, 0), np.repeat(KR, T, 0), 0.5)
    x = 0.5 * (q_lat[0] @ C[0] + q_rope[0] @ KR[0])
    np.testing.assert_allclose(o_lat[0], np.repeat(C, 2, 0), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse[0], x + math.log(T), rtol=1e-14, atol=1e-13)


def test_constant_logit_shift():
    rng = np.random.default_rng(3)
    q_lat, q_rope, C, KR = rand_seq(rng, 1, 1, 50)
    q_rope[0, 0] = [1.0, 0.0, 0.0, 0.0]
    o1, l1 = O.decode_absorbed_seq(q_lat, q_rope, C, KR, 0.3)
    KR2 = KR.copy()
    KR2[:, 0] += 10.0                     # every logit grows by 0.3 * 10
    o2, l2 = O.decode_absorbed_seq(q_lat, q_rope, C, KR2, 0.3)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-14)
    assert l2[0, 0] - l1[0, 0] == pytest.approx(3.0, abs=1e-12)


def test_empty_sequence():
    rng = np.random.default_rng(4)
    q_lat, q_rope, C, KR = rand_seq(rng, 2, 2, 0)
    o_lat, lse = O.decode_absorbed_seq(q_lat, q_rope, C, KR, 0.3, causal=True)
    assert np.all(o_lat == 0) and np.all(np.isneginf(lse))


def test_causal_equals_prefix():
    rng = np.random.default_rng(5)
    q_lat, q_rope, C, KR = rand_seq(rng, 2, 3, 9)
    o, lse = O.decode_absorbed_seq(q_lat, q_rope, C, KR, 0.2, causal=True)
    o0, l0 = O.decode_absorbed_seq(q_lat[:1], q_rope[:1], C[:8], KR[:8], 0.2)
    o1, l1 = O.decode_absorbed_seq(q_lat[1:], q_rope[1:], C, KR, 0.2)
    np.testing.assert_array_equal(o[0], o0[0])
    np.testing.assert_array_equal(o[1], o1[0])
    np.testing.assert_array_equal(lse[0], l0[0])
    assert [O.visible_length(9, 2, s, True) for s in range(2)] == [8, 9]
    assert O.visible_length(9, 2, 0, False) == 9


# ----------------------------------------------------------------------------
# Split-KV log-sum-exp merge
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("cuts", [[0, 7, 50], [0, 1, 2, 3, 50], [0, 25, 25, 50], [0, 50, 60]])
def test_combine_equals_unsplit(cuts):
    rng = np.random.default_rng(6)
    q_lat, q_rope, C, KR = rand_seq(rng, 2, 3, 50)
    n_vis = [50, 50]
    o_ref, l_ref = O.decode_absorbed_seq(q_lat, q_rope, C, KR, 0.4)
    parts = [O.decode_absorbed_partial_seq(q_lat, q_rope, C, KR, 0.4, a, b, n_vis)
             for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = O.combine_partials([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, l_ref, rtol=1e-13, atol=1e-13)


def test_combine_all_empty():
    o, lse = O.combine_partials(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(lse))


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(8).standard_normal((5, 64))
    np.testing.assert_array_equal(O.rope_interleaved(x, np.zeros(5)), x)


def test_rope_unit_vectors_closed_form():
    d, theta, p = 64, 10000.0, 37
    for i in (0, 1, 13, 31):
        e = np.zeros(d)
        e[2 * i] = 1.0
        out = O.rope_interleaved(e, p, theta)
        ang = p * theta ** (-2.0 * i / d)
        expect = np.zeros(d)
        expect[2 * i], expect[2 * i + 1] = math.cos(ang), math.sin(ang)
        np.testing.assert_allclose(out, expect, atol=1e-15)
        e = np.zeros(d)
        e[2 * i + 1] = 1.0
        out = O.rope_interleaved(e, p, theta)
        expect = np.zeros(d)
        expect[2 * i], expect[2 * i + 1] = -math.sin(ang), math.cos(ang)
        np.testing.assert_allclose(out, expect, atol=1e-15)


def test_rope_preserves_pair_norms():
    x = np.random.default_rng(9).standard_normal((7, 64))
    y = O.rope_interleaved(x, np.arange(7) * 1000 + 3)
    np.testing.assert_allclose(np.hypot(y[:, 0::2], y[:, 1::2]), np.hypot(x[:, 0::2], x[:, 1::2]),
                               rtol=1e-13)


def test_rope_relative_position():
    rng = np.random.default_rng(10)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    d1 = O.rope_interleaved(q, 120) @ O.rope_interleaved(k, 100)
    d2 = O.rope_interleaved(q, 5020) @ O.rope_interleaved(k, 5000)
    assert d1 == pytest.approx(d2, rel=1e-10)


# ----------------------------------------------------------------------------
# Paged addressing
# ----------------------------------------------------------------------------

def test_paged_gather_matches_contiguous():
    rng = np.random.default_rng(11)
    T, P = 150, 8
    rows = rng.standard_normal((-(-T // P) * P, 6))
    n_pages = rows.shape[0] // P
    perm = rng.permutation(n_pages + 5)[:n_pages]
    pool = rng.standard_normal((n_pages + 5, P, 6))
    pool[perm] = rows.reshape(n_pages, P, 6)
    np.testing.assert_array_equal(O.gather_paged_rows(pool, perm, T), rows[:T])


# ----------------------------------------------------------------------------
# Planted mistakes: each pin must fail when a plausible error enters the oracle
# ----------------------------------------------------------------------------

def test_planted_mistakes_are_caught():
    g = gold("toy_score.json")
    q_nope, q_rope, c, kr, w_uk = toy_single_row(g)
    q_lat = O.absorb_q(q_nope, w_uk)
    # (1) scale from the latent width, sqrt(d_c + d_r), instead of sqrt(d_nope + d_r)
    _, lse = O.decode_absorbed_seq(q_lat, q_rope, c, kr, 1.0 / math.sqrt(3 + 2))
    assert abs(lse[0, 0] - g["scaled_score"]) > 1e-3
    # (2) the position term dropped from the score
    _, lse = O.decode_absorbed_seq(q_lat, 0 * q_rope, c, kr, O.score_scale(2, 2))
    assert abs(lse[0, 0] - g["scaled_score"]) > 1e-3
    # (3) a wrong index in the absorption (content query read back to front)
    gk = gold("toy_key_absorption.json")
    w = np.array(gk["w_uk_selects_first_two"], float)[None]
    q = np.array(gk["q"], float).reshape(1, 2)
    bad = np.einsum("...hk,hck->...hc", q[..., ::-1], w)[0]
    assert bad.tolist() != gk["q_tilde"]
    # (4) an off-by-one causal mask (query s reads rows < T-S+s): the prefix identity breaks
    rng = np.random.default_rng(5)
    ql, qr, C, KR = rand_seq(rng, 2, 3, 9)
    good, _ = O.decode_absorbed_seq(ql, qr, C, KR, 0.2, causal=True)
    bad_vis = [9 - 2 + s for s in range(2)]
    bad_o, _ = O.decode_absorbed_partial_seq(ql, qr, C, KR, 0.2, 0, 9, bad_vis)
    assert np.abs(bad_o - good).max() > 1e-3
    # (5) RoPE pairing the two halves instead of interleaved neighbours
    def rope_halves(x, pos, theta=10000.0):
        d = x.shape[-1]
        ang = pos * theta ** (-np.arange(0, d, 2) / d)
        a, b = x[: d // 2], x[d // 2:]
        return np.concatenate([a * np.cos(ang) - b * np.sin(ang), a * np.sin(ang) + b * np.cos(ang)])
    e = np.zeros(64)
    e[2] = 1.0
    ang = 37 * 10000.0 ** (-2.0 / 64)
    expect = np.zeros(64)
    expect[2], expect[3] = math.cos(ang), math.sin(ang)
    np.testing.assert_allclose(O.rope_interleaved(e, 37), expect, atol=1e-15)
    assert not np.allclose(rope_halves(e, 37), expect, atol=1e-6)


# ----------------------------------------------------------------------------
# Cache append ([CALC] "계산 재배치의 효과와 한계"; [ANATOMY] section 2)
# ----------------------------------------------------------------------------

def test_append_closed_form_one_pair():
    # d_c = 3, d_r = 2: the only pair has inverse frequency theta^0 = 1, so the row written
    # at position 1 has its k^R turned by exactly 1 radian, whatever theta is; c^KV stays.
    rows, pos = O.append_latent_rows([[1.0, 2.0, 3.0, 1.0, 0.0]], start=1, theta=10000.0, d_r=2)
    assert list(pos) == [1]
    np.testing.assert_array_equal(rows[0, :3], [1.0, 2.0, 3.0])
    np.testing.assert_allclose(rows[0, 3:], [math.cos(1.0), math.sin(1.0)], rtol=0, atol=1e-15)


def test_append_without_rope_keeps_rows_and_counts_positions():
    new = np.arange(3 * 576, dtype=np.float64).reshape(3, 576)
    rows, pos = O.append_latent_rows(new, start=7)
    np.testing.assert_array_equal(rows, new)
    assert list(pos) == [7, 8, 9]


def test_append_all_at_once_equals_one_by_one():
    rng = np.random.default_rng(5)
    new = rng.standard_normal((4, 576))
    rows, pos = O.append_latent_rows(new, start=100, theta=10000.0)
    for s in range(4):
        r1, p1 = O.append_latent_rows(new[s:s + 1], start=100 + s, theta=10000.0)
        np.testing.assert_array_equal(r1[0], rows[s])
        assert p1[0] == pos[s]


def test_append_planted_wrong_position_is_caught():
    # Rotating at start - 1 (an off-by-one in the position) moves the stored k^R.
    new = np.zeros((1, 576))
    new[0, 512] = 1.0
    good, _ = O.append_latent_rows(new, start=3, theta=10000.0)
    bad = new.copy()
    bad[:, 512:] = O.rope_interleaved(bad[:, 512:], np.array([2]), 10000.0)
    assert not np.allclose(good, bad)
    np.testing.assert_allclose(good[0, 512:514], [math.cos(3.0), math.sin(3.0)], atol=1e-15)


# ----------------------------------------------------------------------------
# Pre-fused weights ([CALC] "Query·출력 투영과 합치기")
# ----------------------------------------------------------------------------

def _toy_projections():
    # The pages' toy head 1: d_c = 3, d_k = d_v = 2.  U^K picks the first two latent
    # components ([CALC] "Key 투영을 Query 쪽으로 옮기기"); U^V makes [c0 + c2, c1] ([CALC]
    # "Value 투영을 가중합 뒤로 옮기기").  U^Q (3x2) is not printed; this one takes
    # c^Q = [2, 1, 0] to the pages' content query q = [2, 1].
    u_k = np.array([[[1.0, 0.0], [0.0, 1.0], [0.0, 0.0]]])
    u_v = np.array([[[1.0, 0.0], [0.0, 1.0], [1.0, 0.0]]])
    u_q = np.array([[[1.0, 0.0], [0.0, 1.0], [0.0, 0.0]]])
    return u_q, u_k, u_v


def test_fused_query_weights_reproduce_the_toy_q_tilde():
    u_q, u_k, _ = _toy_projections()
    w = O.fuse_query_weights(u_q, u_k)
    assert w.shape == (1, 3, 3)                       # 3x2 times 2x3
    q_tilde = O.absorb_q_from_latent(np.array([2.0, 1.0, 0.0]), w)
    np.testing.assert_array_equal(q_tilde[0], [2.0, 1.0, 0.0])     # the pages' q~
    assert q_tilde[0] @ np.array([1.0, 2.0, 3.0]) == 4.0           # q~ . c_3 = 4


def test_fused_output_weights_on_the_value_toy():
    # z = [0.8, 1.3, 1.5] ([CALC] value-absorption table) through U^V gives [2.3, 1.3];
    # with a W^O_1 of 2x8 that copies the two head outputs into model columns 0 and 5
    # and their sum into column 7, the fused 3x8 matrix gives head 1's 1x8 contribution.
    _, _, u_v = _toy_projections()
    w_o = np.zeros((1, 2, 8))
    w_o[0, 0, 0] = w_o[0, 1, 5] = w_o[0, 0, 7] = w_o[0, 1, 7] = 1.0
    w = O.fuse_output_weights(u_v, w_o)
    assert w.shape == (1, 3, 8)
    out = O.out_proj_fused(np.array([[0.8, 1.3, 1.5]]), w)
    expect = np.zeros(8)
    expect[0], expect[5], expect[7] = 2.3, 1.3, 3.6
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-15)


def test_fused_forms_equal_the_two_step_products_brute_force():
    rng = np.random.default_rng(9)
    H, d_cq, d_c, d_k, d_model = 3, 5, 4, 2, 6
    w_uq, w_uk = rng.standard_normal((H, d_cq, d_k)), rng.standard_normal((H, d_c, d_k))
    w_uv, w_o = rng.standard_normal((H, d_c, d_k)), rng.standard_normal((H, d_k, d_model))
    c_q, z = rng.standard_normal(d_cq), rng.standard_normal((H, d_c))
    wq, wo = O.fuse_query_weights(w_uq, w_uk), O.fuse_output_weights(w_uv, w_o)
    for h in range(H):                    # scalar loops: q~ = (c_q W_UQ[h]) W_UK[h]^T
        q = [sum(c_q[i] * w_uq[h, i, k] for i in range(d_cq)) for k in range(d_k)]
        qt = [sum(q[k] * w_uk[h, c, k] for k in range(d_k)) for c in range(d_c)]
        np.testing.assert_allclose(O.absorb_q_from_latent(c_q, wq)[h], qt, rtol=1e-12)
    out = np.zeros(d_model)
    for h in range(H):                    # out = sum_h (z_h W_UV[h]) W_O[h]
        v = [sum(z[h, c] * w_uv[h, c, k] for c in range(d_c)) for k in range(d_k)]
        out += [sum(v[k] * w_o[h, k, j] for k in range(d_k)) for j in range(d_model)]
    np.testing.assert_allclose(O.out_proj_fused(z, wo), out, rtol=1e-12)
    np.testing.assert_allclose(O.out_proj_heads(O.out_proj_uv(z, w_uv), w_o), out, rtol=1e-12)


def test_fused_planted_transpose_is_caught():
    # Multiplying W_UQ by W_UK without the transpose (a wrong index) changes q~.
    rng = np.random.default_rng(3)
    w_uq, w_uk = rng.standard_normal((1, 4, 4)), rng.standard_normal((1, 4, 4))
    c_q = rng.standard_normal(4)
    good = O.absorb_q_from_latent(c_q, O.fuse_query_weights(w_uq, w_uk))
    bad = np.einsum("i,hic->hc", c_q, np.einsum("hik,hkc->hic", w_uq, w_uk))
    assert not np.allclose(good, bad)


# ----------------------------------------------------------------------------
# FP8 latent cache: the E4M3 format of the OCP 8-bit floating point specification
# (bias 7, subnormals at exponent 0, no infinities, S.1111.111 NaN, largest 448), a
# power-of-two scale per token over the 512 latent values
# ----------------------------------------------------------------------------

def test_e4m3_closed_forms():
    v = O.e4m3_decode
    assert v(0x7E) == 448.0                       # S.1111.110: (1 + 6/8) * 2^8
    assert v(0x01) == 2.0 ** -9                   # smallest subnormal: 1/8 * 2^-6
    assert v(0x07) == 7 * 2.0 ** -9               # largest subnormal
    assert v(0x08) == 2.0 ** -6                   # smallest normal
    assert v(0x38) == 1.0                         # exponent field 7 = bias
    assert v(0x3C) == 1.5 and v(0xBC) == -1.5
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    assert v(0x00) == 0.0 and np.signbit(v(0x80))
    pos = v(np.arange(0x7F))
    assert pos.size == 127 and np.all(np.diff(pos) > 0)       # 127 distinct, increasing
    # every normal binade holds 8 values spaced 2^(e-10)
    for e in range(1, 16):
        b = v(np.arange(8 * e, 8 * e + 8)) if 8 * e + 8 <= 0x7F else None
        if b is not None:
            assert np.allclose(np.diff(b), 2.0 ** (e - 10))


def test_e4m3_encode_round_trip_and_ties():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)     # -0.0 <-> 0x80 included
    e = O.e4m3_encode
    assert e(1.0625) == 0x38 and e(1.1875) == 0x3A          # ties to the even mantissa
    assert e(2.0 ** -10) == 0x00 and e(1.5 * 2.0 ** -10) == 0x01   # below the smallest subnormal
    assert e(464.0) == 0x7E and e(500.0) == 0x7E and e(1e30) == 0x7E and e(-1e30) == 0xFE   # saturation
    assert e(-2.0 ** -11) == 0x80


def test_e4m3_encode_matches_the_torch_float8_type():
    # torch.float8_e4m3fn rounds to nearest even (it does not saturate, so the
    # comparison stays within +-448).
    import torch
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 30, 20000), rng.normal(0, 0.01, 5000), rng.uniform(-448, 448, 5000)])
    x = np.clip(x, -448, 448)
    ref = torch.tensor(x, dtype=torch.float64).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x), ref)


def test_fp8_row_scale_is_the_least_power_of_two():
    rng = np.random.default_rng(4)
    for _ in range(200):
        row = rng.normal(0, 10 ** rng.uniform(-6, 4), 512)
        s = O.fp8_row_scale(row)
        assert math.frexp(s)[0] == 0.5                        # a power of two
        amax = np.abs(row).max()
        assert amax / s <= 448.0 < amax / (s / 2)
    assert O.fp8_row_scale(np.zeros(512)) == 1.0
    assert O.fp8_row_scale([448.0]) == 1.0 and O.fp8_row_scale([449.0]) == 2.0
    assert O.fp8_row_scale([224.0]) == 0.5
    assert O.fp8_row_scale([1e9]) == 2.0 ** 15                 # the exponent's upper clamp
    assert O.e4m3_encode(1e9 / 2.0 ** 15) == 0x7E              # ... and the row saturates


def test_fp8_quantize_error_bound_and_rope_untouched():
    rng = np.random.default_rng(5)
    rows = rng.normal(0, 1, (40, 576))
    rows[3, :512] = 0.0
    codes, kr, scales = O.quantize_fp8_rows(rows)
    assert codes.dtype == np.uint8 and codes.shape == (40, 512)
    assert np.array_equal(kr, rows[:, 512:])
    back = O.dequantize_fp8_rows(codes, kr, scales)
    err = np.abs(back[:, :512] - rows[:, :512])
    # nearest rounding: half a step of the binade (2^(e-4) relative) for normals, half
    # the subnormal step (2^-10 * scale) below 2^-6 * scale
    bound = np.maximum(np.abs(rows[:, :512]) * 2.0 ** -4, 2.0 ** -10 * scales[:, None])
    assert np.all(err <= bound)
    assert np.all(back[3, :512] == 0.0) and scales[3] == 1.0
    # values already on the grid come back exactly (the scale may halve when the row's
    # maximum rounded down onto 224 * scale)
    codes2, kr2, scales2 = O.quantize_fp8_rows(back)
    assert np.array_equal(O.dequantize_fp8_rows(codes2, kr2, scales2), back)
    assert np.all((scales2 == scales) | (scales2 == scales / 2))


def test_fp8_planted_mistakes_are_caught():
    # A plain truncation instead of nearest rounding, and a scale that is not the least
    # power of two, both break the pins above.
    pos = O.e4m3_decode(np.arange(0x7F))
    trunc = lambda a: np.searchsorted(pos, a, side="right") - 1
    assert trunc(1.0625 + 0.06) != O.e4m3_encode(1.0625 + 0.06)
    loose = lambda row: 2.0 * O.fp8_row_scale(row)
    row = np.array([300.0])
    assert not (np.abs(row).max() / loose(row) > 224.0)
