"""Pins for the fp64 oracle: each check rests on something other than the oracle itself
(a closed form, an exact identity, brute force, or the arithmetic printed on the pages).
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import mla_oracle as M

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand_case(rng, n_h=3, L=7, scale_w=1.0 / math.sqrt(512)):
    q = rng.standard_normal((n_h, 192))
    c = rng.standard_normal((L, 512))
    kr = rng.standard_normal((L, 64))
    wk = rng.standard_normal((n_h, 128, 512)) * scale_w
    wv = rng.standard_normal((n_h, 128, 512)) * scale_w
    return q, c, kr, wk, wv


# ------------------------------- RoPE ---------------------------------------------
def test_rope_zero_position_is_identity():
    x = np.random.default_rng(1).standard_normal((5, 64))
    np.testing.assert_array_equal(M.rope(x, 0), x)


def test_rope_preserves_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((9, 64))
    pos = rng.integers(0, 131072, size=9)
    y = M.rope(x, pos)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_closed_form_unit_vectors():
    # e_0 at position 1 rotates by exactly 1 radian into the (0, 32) plane.
    e0 = np.zeros(64); e0[0] = 1.0
    y = M.rope(e0, 1)
    assert y[0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert y[32] == pytest.approx(math.sin(1.0), abs=1e-15)
    assert np.count_nonzero(np.abs(y) > 1e-15) == 2
    # e_32 goes the other way: x'_0 = -sin, x'_32 = cos.
    e32 = np.zeros(64); e32[32] = 1.0
    y = M.rope(e32, 1)
    assert y[0] == pytest.approx(-math.sin(1.0), abs=1e-15)
    assert y[32] == pytest.approx(math.cos(1.0), abs=1e-15)
    # pair i = 5 turns with frequency 10000^(-10/64).
    e5 = np.zeros(64); e5[5] = 1.0
    p = 12345
    ang = p * 10000.0 ** (-10.0 / 64.0)
    y = M.rope(e5, p)
    assert y[5] == pytest.approx(math.cos(ang), abs=1e-12)
    assert y[37] == pytest.approx(math.sin(ang), abs=1e-12)


def test_rope_relative_position_invariance():
    # Shifting the query and every key position by the same amount leaves the
    # attention result unchanged (RoPE encodes only relative position).
    rng = np.random.default_rng(3)
    q, c, kr_raw, wk, wv = _rand_case(rng, n_h=2, L=6)
    t = np.arange(6)
    base = M.attend_explicit(q, c, M.rope(kr_raw, t), wk, wv, pos_q=5)
    for delta in (1, 1000, 100000):
        sh = M.attend_explicit(q, c, M.rope(kr_raw, t + delta), wk, wv, pos_q=5 + delta)
        np.testing.assert_allclose(sh["o"], base["o"], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(sh["lse"], base["lse"], rtol=1e-9)


# --------------------------- attention identities ---------------------------------
def test_absorbed_matches_explicit_bruteforce_sizes():
    rng = np.random.default_rng(4)
    for n_h, L in [(1, 1), (2, 3), (4, 8), (3, 5)]:
        q, c, kr, wk, wv = _rand_case(rng, n_h=n_h, L=L)
        a = M.attend_explicit(q, c, kr, wk, wv, pos_q=L - 1)
        b = M.attend_absorbed(q, c, kr, wk, wv, pos_q=L - 1)
        for k in ("o", "o_lat", "lse"):
            np.testing.assert_allclose(a[k], b[k], rtol=1e-12, atol=1e-13)


def test_latent_form_matches_explicit_bruteforce_sizes():
    # the absorbed query built by hand reproduces the explicit form's o_lat and lse
    rng = np.random.default_rng(41)
    for n_h, L, pos in [(1, 1, 0), (2, 3, 2), (4, 8, 100), (3, 5, 131071)]:
        q, c, kr, wk, wv = _rand_case(rng, n_h=n_h, L=L)
        a = M.attend_explicit(q, c, kr, wk, wv, pos_q=pos)
        q_lat = np.concatenate([np.einsum("hd,hdj->hj", q[:, :128], wk), M.rope(q[:, 128:], pos)], axis=1)
        b = M.attend_latent(q_lat, np.concatenate([c, kr], axis=1))
        np.testing.assert_allclose(b["o_lat"], a["o_lat"], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(b["lse"], a["lse"], rtol=1e-12, atol=1e-13)


def test_latent_form_scalar_bruteforce():
    rng = np.random.default_rng(42)
    q_lat = rng.standard_normal((2, 576)) * 3.0
    rows = rng.standard_normal((4, 576))
    r = M.attend_latent(q_lat, rows)
    scale = 1.0 / math.sqrt(192.0)
    for h in range(2):
        s = [sum(q_lat[h, d] * rows[t, d] for d in range(576)) * scale for t in range(4)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        for j in (0, 7, 300, 511):
            assert r["o_lat"][h, j] == pytest.approx(sum(e[t] / z * rows[t, j] for t in range(4)), rel=1e-12, abs=1e-14)
        assert r["lse"][h] == pytest.approx(m + math.log(z), rel=1e-13)


def _scalar_loop_attention(q, c, kr, wk, wv, pos_q, scale):
    """Brute force with Python scalars only (no NumPy linear algebra)."""
    n_h, L = q.shape[0], c.shape[0]
    out = []
    for h in range(n_h):
        qr = [0.0] * 64
        for i in range(32):
            th = pos_q * 10000.0 ** (-2.0 * i / 64.0)
            qr[i] = q[h, 128 + i] * math.cos(th) - q[h, 160 + i] * math.sin(th)
            qr[32 + i] = q[h, 160 + i] * math.cos(th) + q[h, 128 + i] * math.sin(th)
        s = []
        vs = []
        for t in range(L):
            acc = 0.0
            for d in range(128):
                k_d = sum(wk[h, d, j] * c[t, j] for j in range(512))
                acc += q[h, d] * k_d
            for d in range(64):
                acc += qr[d] * kr[t, d]
            s.append(acc * scale)
            vs.append([sum(wv[h, d, j] * c[t, j] for j in range(512)) for d in range(128)])
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        o = [sum(e[t] / z * vs[t][d] for t in range(L)) for d in range(128)]
        out.append((o, m + math.log(z)))
    return out


def test_explicit_matches_scalar_bruteforce():
    rng = np.random.default_rng(5)
    q, c, kr, wk, wv = _rand_case(rng, n_h=2, L=3)
    r = M.attend_explicit(q, c, kr, wk, wv, pos_q=7)
    bf = _scalar_loop_attention(q, c, kr, wk, wv, 7, M.default_scale())
    for h, (o, lse) in enumerate(bf):
        np.testing.assert_allclose(r["o"][h], o, rtol=1e-11, atol=1e-13)
        assert r["lse"][h] == pytest.approx(lse, rel=1e-12)


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(6)
    q, c, kr, wk, wv = _rand_case(rng, n_h=4, L=50)
    r = M.attend_explicit(q * 5, c, kr, wk, wv, pos_q=49, return_p=True)
    assert np.all(r["p"] >= 0)
    np.testing.assert_allclose(r["p"].sum(axis=1), 1.0, atol=1e-12)


def test_length_one_returns_that_tokens_value():
    rng = np.random.default_rng(7)
    q, c, kr, wk, wv = _rand_case(rng, n_h=4, L=1)
    r = M.attend_explicit(q, c, kr, wk, wv, pos_q=0)
    for h in range(4):
        np.testing.assert_allclose(r["o"][h], wv[h] @ c[0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(r["o_lat"][h], c[0], rtol=1e-13, atol=1e-14)


def test_constant_cache_returns_projected_row():
    rng = np.random.default_rng(8)
    q, c, kr, wk, wv = _rand_case(rng, n_h=3, L=9)
    c[:] = c[0]
    kr[:] = kr[0]
    r = M.attend_explicit(q, c, kr, wk, wv, pos_q=8)
    for h in range(3):
        np.testing.assert_allclose(r["o"][h], wv[h] @ c[0], rtol=1e-12, atol=1e-14)
        assert r["lse"][h] == pytest.approx(
            (np.concatenate([wk[h] @ c[0], kr[0]]) @ np.concatenate(
                [q[h, :128], M.rope(q[h, 128:], 8)])) * M.default_scale() + math.log(9), rel=1e-12)


def test_zero_query_gives_uniform_weights():
    rng = np.random.default_rng(9)
    _, c, kr, wk, wv = _rand_case(rng, n_h=2, L=33)
    q = np.zeros((2, 192))
    r = M.attend_explicit(q, c, kr, wk, wv, pos_q=32)
    np.testing.assert_allclose(r["o_lat"], np.broadcast_to(c.mean(axis=0), (2, 512)), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["lse"], math.log(33), rtol=1e-14)


def test_two_token_closed_form_pins_scale_and_orientation():
    # Token 0 is all zeros; token 1 has latent e_k and RoPE key e_j.
    # s_0 = 0 and s_1 = scale·(q^C·W_UK[h][:, k] + q^R'_j), so p_1 = sigmoid(s_1),
    # o = p_1·W_UV[h][:, k] and o^lat = p_1·e_k.
    rng = np.random.default_rng(10)
    n_h, k, j = 2, 37, 11
    wk = rng.standard_normal((n_h, 128, 512)) / math.sqrt(512)
    wv = rng.standard_normal((n_h, 128, 512)) / math.sqrt(512)
    q = rng.standard_normal((n_h, 192))
    c = np.zeros((2, 512)); c[1, k] = 1.0
    kr = np.zeros((2, 64)); kr[1, j] = 1.0
    r = M.attend_explicit(q, c, kr, wk, wv, pos_q=0)     # position 0: no rotation
    scale = 1.0 / math.sqrt(192.0)
    for h in range(n_h):
        s1 = scale * (q[h, :128] @ wk[h][:, k] + q[h, 128 + j])
        p1 = 1.0 / (1.0 + math.exp(-s1))
        np.testing.assert_allclose(r["o"][h], p1 * wv[h][:, k], rtol=1e-12, atol=1e-15)
        assert r["o_lat"][h, k] == pytest.approx(p1, rel=1e-12)
        assert r["lse"][h] == pytest.approx(math.log(1.0 + math.exp(s1)), rel=1e-12)


def test_empty_context():
    rng = np.random.default_rng(11)
    q, c, kr, wk, wv = _rand_case(rng, n_h=2, L=0)
    r = M.attend_explicit(q, c, kr, wk, wv, pos_q=0)
    assert np.all(r["o"] == 0) and np.all(r["o_lat"] == 0)
    assert np.all(np.isneginf(r["lse"]))


def test_merge_of_disjoint_parts_equals_whole():
    rng = np.random.default_rng(12)
    q, c, kr, wk, wv = _rand_case(rng, n_h=3, L=40)
    whole = M.attend_explicit(q, c, kr, wk, wv, pos_q=39)
    cuts = [0, 7, 7, 23, 40]          # includes an empty part
    parts = [M.attend_explicit(q, c[a:b], kr[a:b], wk, wv, pos_q=39) for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = M.merge_partials(np.stack([p["o_lat"] for p in parts]), np.stack([p["lse"] for p in parts]))
    np.testing.assert_allclose(o, whole["o_lat"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, whole["lse"], rtol=1e-13)
    # all parts empty → zero output, -inf lse
    o0, l0 = M.merge_partials(np.zeros((2, 3, 512)), np.full((2, 3), -np.inf))
    assert np.all(o0 == 0) and np.all(np.isneginf(l0))


# --------------------------- cache-size arithmetic --------------------------------
def test_cache_size_matches_the_pages():
    g = json.load(open(os.path.join(HERE, "golden", "cache_arithmetic.json")))
    assert M.mla_cache_elements(g["d_c"], g["d_rope"], 1) == g["row_elements"] == M.D_ROW
    assert M.mha_cache_elements(g["n_heads"], M.D_H, 1) == 32768
    assert M.gqa_equivalent_groups(g["d_c"], g["d_rope"], M.D_H) == g["gqa_groups"]
    b1 = M.mla_cache_bytes(g["d_c"], g["d_rope"], g["layers"], g["context_tokens"], 1,
                           g["avg_bits_per_element"]) / 1e9
    b64 = M.mla_cache_bytes(g["d_c"], g["d_rope"], g["layers"], g["context_tokens"], 64,
                            g["avg_bits_per_element"]) / 1e9
    assert abs(b1 - g["cache_gb_batch1_printed"]) <= g["printed_precision_gb"]["batch1"]
    assert abs(b64 - g["cache_gb_batch64_printed"]) <= g["printed_precision_gb"]["batch64"]


# ----------------------------- writing the cache ----------------------------------
def _append_case(rng, T=4, d=96):
    h = rng.standard_normal((T, d))
    w_dkv = rng.standard_normal((512, d)) / math.sqrt(d)
    w_kr = rng.standard_normal((64, d)) / math.sqrt(d)
    return h, w_dkv, w_kr


def test_cache_rows_of_basis_states_are_weight_columns():
    # h = e_j: the latent is column j of W_DKV exactly; at position 0 the key is column j
    # of W_KR unrotated, at position p it is that column turned by RoPE.
    rng = np.random.default_rng(40)
    _, w_dkv, w_kr = _append_case(rng)
    for j in (0, 17, 95):
        e = np.zeros((1, 96)); e[0, j] = 1.0
        r0 = M.cache_rows(e, w_dkv, w_kr, [0])
        np.testing.assert_array_equal(r0[0, :512], w_dkv[:, j])
        np.testing.assert_array_equal(r0[0, 512:], w_kr[:, j])
        r = M.cache_rows(e, w_dkv, w_kr, [777])
        np.testing.assert_array_equal(r[0, :512], w_dkv[:, j])
        np.testing.assert_allclose(r[0, 512:], M.rope(w_kr[:, j], 777), rtol=0, atol=1e-15)
        assert not np.allclose(r[0, 512:], w_kr[:, j])


def test_cache_rows_scalar_bruteforce():
    rng = np.random.default_rng(41)
    h, w_dkv, w_kr = _append_case(rng, T=2, d=8)
    pos = [3, 40]
    got = M.cache_rows(h, w_dkv, w_kr, pos)
    for t in range(2):
        for i in range(512):
            assert got[t, i] == pytest.approx(sum(w_dkv[i, j] * h[t, j] for j in range(8)), rel=1e-12, abs=1e-14)
        raw = [sum(w_kr[i, j] * h[t, j] for j in range(8)) for i in range(64)]
        for i in range(32):
            ang = pos[t] * 10000.0 ** (-i / 32.0)
            assert got[t, 512 + i] == pytest.approx(raw[i] * math.cos(ang) - raw[i + 32] * math.sin(ang), abs=1e-12)
            assert got[t, 544 + i] == pytest.approx(raw[i + 32] * math.cos(ang) + raw[i] * math.sin(ang), abs=1e-12)


def test_written_keys_attend_by_relative_position():
    # Rows written at positions t + delta, read by a query at L - 1 + delta: the
    # attention result does not depend on delta, so each key is turned by its own
    # position, the same way as the query.
    rng = np.random.default_rng(42)
    L, d = 6, 32
    h, w_dkv, w_kr = _append_case(rng, T=L, d=d)
    q, _, _, wk, wv = _rand_case(rng, n_h=2, L=L)
    ref = None
    for delta in (0, 9, 50000):
        rows = M.cache_rows(h, w_dkv, w_kr, np.arange(L) + delta)
        out = M.attend_explicit(q, rows[:, :512], rows[:, 512:], wk, wv, pos_q=L - 1 + delta)
        if ref is None:
            ref = out
        else:
            np.testing.assert_allclose(out["o"], ref["o"], rtol=1e-9, atol=1e-12)
            np.testing.assert_allclose(out["lse"], ref["lse"], rtol=1e-9)


def test_cache_rows_are_linear_in_the_hidden_state():
    rng = np.random.default_rng(43)
    h, w_dkv, w_kr = _append_case(rng, T=3)
    h2 = rng.standard_normal(h.shape)
    pos = [5, 6, 1000]
    lhs = M.cache_rows(2.5 * h - h2, w_dkv, w_kr, pos)
    rhs = 2.5 * M.cache_rows(h, w_dkv, w_kr, pos) - M.cache_rows(h2, w_dkv, w_kr, pos)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-10, atol=1e-12)


# ----------------------------- YaRN frequencies ------------------------------------
YARN = dict(scale=40.0, alpha=1.0, beta=32.0, original_max_pos=4096)   # the pages' parameters, 4K pre-training


def test_yarn_scale_one_is_plain_rope():
    f = M.yarn_inv_freq(64, 10000.0, 1.0, 1.0, 32.0, 4096)
    np.testing.assert_array_equal(f, 10000.0 ** (-np.arange(32) / 32.0))
    x = np.random.default_rng(50).standard_normal((3, 64))
    np.testing.assert_array_equal(M.rope(x, [1, 700, 90000], inv_freq=f), M.rope(x, [1, 700, 90000]))


def test_yarn_bands_for_the_pages_parameters():
    # Pair i turns r_i = 4096 · 10000^(-i/32) / (2π) times over the 4K context:
    # r_10 = 36.7 and r_11 = 27.5 (β = 32 lies between), r_22 = 1.16 and r_23 = 0.87
    # (α = 1 lies between). So pairs 0..10 keep their frequency, 23..31 are slowed by
    # exactly 40, and 11..22 lie strictly in between.
    plain = 10000.0 ** (-np.arange(32) / 32.0)
    f = M.yarn_inv_freq(64, 10000.0, **YARN)
    np.testing.assert_array_equal(f[:11], plain[:11])
    np.testing.assert_allclose(f[23:], plain[23:] / 40.0, rtol=1e-15)
    mid = f[11:23] / plain[11:23]
    assert np.all((mid > 1 / 40.0) & (mid < 1.0))
    assert np.all(np.diff(f / plain) <= 1e-15)   # the slowdown grows with the wavelength


def test_yarn_frequency_of_a_ramp_pair():
    # pair 16: θ = 0.01, r = 40.96 / (2π) = 6.51899, ramp (r - 1) / 31 = 0.178032,
    # θ' = 0.01 · (0.178032 + 0.821968 / 40) = 0.00198581
    f = M.yarn_inv_freq(64, 10000.0, **YARN)
    assert f[16] == pytest.approx(0.0019858103, rel=1e-7)


def test_yarn_keys_attend_by_relative_position():
    rng = np.random.default_rng(51)
    L, d = 5, 32
    f = M.yarn_inv_freq(64, 10000.0, **YARN)
    h, w_dkv, w_kr = _append_case(rng, T=L, d=d)
    q, _, _, wk, wv = _rand_case(rng, n_h=2, L=L)
    outs = []
    for delta in (0, 3000, 150000):
        rows = M.cache_rows(h, w_dkv, w_kr, np.arange(L) + delta, inv_freq=f)
        outs.append(M.attend_explicit(q, rows[:, :512], rows[:, 512:], wk, wv, pos_q=L - 1 + delta, inv_freq=f))
    for o in outs[1:]:
        np.testing.assert_allclose(o["o"], outs[0]["o"], rtol=1e-9, atol=1e-12)


# ------------------------------ several new tokens ---------------------------------
def _multi_case(rng, T=3, L=9, n_h=2):
    _, c, kr, wk, wv = _rand_case(rng, n_h=n_h, L=L)
    q = rng.standard_normal((T, n_h, 192))
    return q, c, kr, wk, wv


def test_multi_token_last_query_is_the_single_token_decode():
    rng = np.random.default_rng(60)
    q, c, kr, wk, wv = _multi_case(rng)
    out = M.attend_multi(q, c, kr, wk, wv, T=3)
    single = M.attend_explicit(q[2], c, kr, wk, wv, pos_q=c.shape[0] - 1)
    np.testing.assert_allclose(out["o"][2], single["o"], rtol=1e-12, atol=1e-14)
    one = M.attend_multi(q[2:], c, kr, wk, wv, T=1)
    np.testing.assert_allclose(one["o"][0], single["o"], rtol=1e-12, atol=1e-14)


def test_multi_token_queries_do_not_see_later_tokens():
    # query j sees tokens 0 .. L - T + j: changing the tokens after that position changes
    # nothing for it, and changing the token at that position does
    rng = np.random.default_rng(61)
    q, c, kr, wk, wv = _multi_case(rng, T=4, L=10)
    base = M.attend_multi(q, c, kr, wk, wv, T=4)
    for j in range(4):
        p = 10 - 4 + j
        c2, kr2 = c.copy(), kr.copy()
        c2[p + 1:] += 5.0
        kr2[p + 1:] -= 3.0
        out = M.attend_multi(q, c2, kr2, wk, wv, T=4)
        np.testing.assert_array_equal(out["o"][j], base["o"][j])
        c3 = c.copy()
        c3[p] += 1.0
        assert not np.allclose(M.attend_multi(q, c3, kr, wk, wv, T=4)["o"][j], base["o"][j])


def test_multi_token_positions_and_empty_queries():
    # with L < T the first T - L queries see no token; the others sit at 0, 1, ...
    rng = np.random.default_rng(62)
    q, c, kr, wk, wv = _multi_case(rng, T=4, L=2)
    out = M.attend_multi(q, c, kr, wk, wv, T=4)
    assert np.all(out["o"][:2] == 0) and np.all(np.isneginf(out["lse"][:2]))
    # query 2 sees token 0 alone: its output is that token's value, W_UV · c_0
    np.testing.assert_allclose(out["o"][2], np.einsum("hdj,j->hd", wv, c[0]), rtol=1e-12)
    np.testing.assert_allclose(out["o_lat"][2], np.broadcast_to(c[0], (2, 512)), rtol=1e-12)
