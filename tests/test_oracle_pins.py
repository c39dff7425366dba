"""Pins of the CPU oracle against closed forms, brute force and invariants (no GPU).

Each test pins one oracle function to something other than itself: a closed
form, a hand-derived value, a brute-force loop on a tiny input, or an
invariant that a dropped term, wrong sign or transposed operand would break.
"""
import math

import numpy as np
import pytest

import synthetic as syn
from oracle import attention, cache, quant, rotation


# ---------------------------------------------------------------- Hadamard
@pytest.mark.parametrize("d", [1, 2, 4, 8, 64, 128])
def test_hadamard_closed_form(d):
    h = rotation.sylvester_hadamard(d)
    for i in range(d):
        for j in range(d):
            assert h[i, j] == (-1) ** bin(i & j).count("1") / math.sqrt(d)
    assert np.abs(h @ h - np.eye(d)).max() < 1e-13  # symmetric and orthonormal


def test_hadamard_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        rotation.sylvester_hadamard(12)


# ---------------------------------------------------------------- bit reversal
def test_bit_reversal_d8():
    assert list(rotation.bit_reversal(8)) == [0, 4, 2, 6, 1, 5, 3, 7]


@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_bit_reversal_involution(d):
    p = rotation.bit_reversal_matrix(d)
    assert np.array_equal(p @ p, np.eye(d))
    assert np.array_equal(p, p.T)
    x = np.arange(d, dtype=np.float64) * 3 + 1
    br = rotation.bit_reversal(d)
    assert np.array_equal(x @ p, x[br])  # (x P)_j = x_{br(j)}


# ---------------------------------------------------------------- covariances and eigenbasis
def test_query_covariance_closed_form():
    q = np.array([[1.0, 0.0], [0.0, 2.0], [1.0, 1.0]])
    # (1/3) * ([1,0;0,0] + [0,0;0,4] + [1,1;1,1])
    assert np.allclose(rotation.query_covariance(q), np.array([[2.0, 1.0], [1.0, 5.0]]) / 3, atol=0, rtol=1e-15)


def test_score_covariance_single_token_is_outer_product():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 1, 4))
    k = rng.standard_normal((1, 1, 4))
    v = rng.standard_normal((1, 1, 4))
    assert np.allclose(rotation.score_covariance(q, k, v), np.outer(v[0, 0], v[0, 0]), rtol=1e-14, atol=1e-15)


def test_score_covariance_zero_query_causal_means():
    # q = 0 makes every causal softmax row uniform over the visible prefix
    rng = np.random.default_rng(8)
    t, d = 3, 4
    q = np.zeros((t, 2, d))
    k = rng.standard_normal((t, 1, d))
    v = rng.standard_normal((t, 1, d))
    rows = [v[0, 0], (v[0, 0] + v[1, 0]) / 2, (v[0, 0] + v[1, 0] + v[2, 0]) / 3]
    want = sum(np.outer(r, r) for r in rows) / t  # both query heads see the same rows
    assert np.allclose(rotation.score_covariance(q, k, v), want, rtol=1e-13, atol=1e-14)


def test_score_covariance_brute_force_small():
    rng = np.random.default_rng(9)
    t, hq, hkv, d = 4, 2, 1, 3
    q = rng.standard_normal((t, hq, d))
    k = rng.standard_normal((t, hkv, d))
    v = rng.standard_normal((t, hkv, d))
    want = np.zeros((d, d))
    for h in range(hq):
        for i in range(t):
            logits = [sum(q[i, h, c] * k[j, 0, c] for c in range(d)) / math.sqrt(d) for j in range(i + 1)]
            mx = max(logits)
            e = [math.exp(x - mx) for x in logits]
            o = [sum(e[j] / sum(e) * v[j, 0, c] for j in range(i + 1)) for c in range(d)]
            for a in range(d):
                for b in range(d):
                    want[a, b] += o[a] * o[b]
    want /= t * hq
    assert np.allclose(rotation.score_covariance(q, k, v), want, rtol=1e-12, atol=1e-14)


def test_eigenbasis_diagonal_is_sorted_permutation():
    u = rotation.eigenbasis(np.diag([3.0, 1.0, 2.0]))
    assert np.array_equal(u, np.array([[1.0, 0, 0], [0, 0, 1.0], [0, 1.0, 0]]))


def test_eigenbasis_random_spd():
    rng = np.random.default_rng(10)
    a = rng.standard_normal((16, 16))
    c = a @ a.T / 16 + np.diag(rng.uniform(0.1, 1, 16))
    u = rotation.eigenbasis(c)
    lam = np.diag(u.T @ c @ u)
    assert np.all(np.diff(lam) <= 1e-12)  # descending
    assert np.abs(u.T @ c @ u - np.diag(lam)).max() < 1e-12
    piv = np.argmax(np.abs(u), axis=0)
    assert np.all(u[piv, np.arange(16)] > 0)  # sign rule


# ---------------------------------------------------------------- composite rotation
def test_rotation_identity_u_is_hadamard_times_bitrev():
    d = 64
    r = rotation.composite_rotation(np.eye(d))
    assert np.array_equal(r, rotation.sylvester_hadamard(d) @ rotation.bit_reversal_matrix(d))
    # column j of H P is column br(j) of H
    assert np.array_equal(r, rotation.sylvester_hadamard(d)[:, rotation.bit_reversal(d)])


@pytest.mark.parametrize("wl", [syn.tiny(), syn.batch1_32k()], ids=lambda w: w.name)
def test_layer_fixture_rotations_orthogonal(wl):
    s = wl.shape
    q = syn.queries(wl, 0, 64, calib=True)
    k, v = syn.kv_tokens(wl, 0, 64, calib=True)
    fx = rotation.layer_fixture(q, k, v)
    for key in ("R_K64", "R_V64"):
        r = fx[key]
        assert r.shape == (s.head_dim, s.head_dim)
        assert np.abs(r @ r.T - np.eye(s.head_dim)).max() < 1e-12
    # the product's first factor is the eigenbasis of C_Q: R P^T H^T = U_Q
    d = s.head_dim
    back = fx["R_K64"] @ rotation.bit_reversal_matrix(d).T @ rotation.sylvester_hadamard(d).T
    assert np.abs(back - fx["U_Q"]).max() < 1e-12
    assert fx["clip_K"] > 0 and fx["clip_V"] > 0


def test_clip_threshold_percentile_closed_form():
    x = np.arange(1001, dtype=np.float64)[:, None] - 500.0  # |x| takes 0..500, each twice except 0
    r = np.array([[1.0]])
    # sorted |x|: 0, 1,1, 2,2, ..., 500,500 (1001 values); 99.9th pct at rank 999 -> value 500
    assert rotation.clip_threshold(x, r) == 500.0
    x2 = np.arange(1001, dtype=np.float64)[:, None]
    assert rotation.clip_threshold(x2, np.array([[-1.0]])) == pytest.approx(999.0, rel=1e-14)
    # rank 999.999 of 0..1000 under linear interpolation
    assert rotation.clip_threshold(x2, np.array([[1.0]]), pct=99.95) == pytest.approx(999.5, rel=1e-14)


# ---------------------------------------------------------------- BF16 rounding
def _bf16_via_f32_bits(x):
    """Independent route for float32-representable values: integer round-to-nearest-even on the bits."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def test_bf16_round_hand_values():
    f = quant.bf16_round
    assert f(1.0) == 1.0
    assert f(1 + 2.0 ** -8) == 1.0                         # tie -> even
    assert f(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6           # tie -> even (up)
    assert f(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7  # just above the tie
    assert f(-3.0) == -3.0
    assert f(2.0 ** -133) == 2.0 ** -133                    # smallest subnormal
    assert f(2.0 ** -134) == 0.0                            # tie -> even (zero)
    assert f(3 * 2.0 ** -134) == 2.0 ** -132                # tie -> even (two quanta)
    assert f(0.0) == 0.0


def test_bf16_round_matches_bit_route():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32).astype(np.float64)
    assert np.array_equal(quant.bf16_round(x), _bf16_via_f32_bits(x))


# ---------------------------------------------------------------- quantiser
def test_quantizer_on_grid_round_trip():
    rng = np.random.default_rng(12)
    for _ in range(200):
        z = quant.bf16_round(rng.standard_normal() * 4)
        s = quant.bf16_round(abs(rng.standard_normal()) + 0.05)
        codes = rng.integers(0, 4, size=32)
        codes[rng.integers(0, 32)] = 0
        codes[rng.integers(0, 32)] = 3
        if codes.min() != 0 or codes.max() != 3:
            continue
        y = z + codes * s
        c, sc, zz, _, _ = quant.quantize_groups(y[None, :], 32)
        assert sc[0, 0] == s and zz[0, 0] == z
        assert np.array_equal(c[0], codes)
        assert np.array_equal(quant.dequantize(c, sc, zz, 32)[0], y)


def test_quantizer_brute_force_nearest_level_and_bounds():
    rng = np.random.default_rng(13)
    y = rng.standard_normal((500, 64)) * rng.uniform(0.1, 10, (500, 1))
    c = 2.5
    y = np.clip(y, -c, c)
    codes, scale, zero, mn, rng3 = quant.quantize_groups(y, 32)
    assert codes.dtype == np.uint8 and codes.max() <= 3
    yg = y.reshape(500, 2, 32)
    cg = codes.reshape(500, 2, 32)
    # brute force: the code picks the nearest of the 4 levels of its group (clamped range)
    levels = zero[..., None] + np.arange(4)[None, None, :] * scale[..., None]  # [500, 2, 4]
    dist = np.abs(yg[..., None] - levels[:, :, None, :])                       # [500, 2, 32, 4]
    best = np.argmin(dist, axis=-1)
    assert np.array_equal(best, cg)
    # error bound |y - y_hat| <= s/2 + |mn - z| + 3 |rng3 - s|
    yhat = quant.dequantize(codes, scale, zero, 32).reshape(500, 2, 32)
    bound = scale / 2 + np.abs(mn - zero) + 3 * np.abs(rng3 - scale)
    assert np.all(np.abs(yg - yhat) <= bound[..., None] * (1 + 1e-12))
    # clip bounds and both extreme codes present in ordinary groups
    assert np.all(mn >= -c) and np.all(mn + 3 * rng3 <= c + 1e-12)
    assert np.all(cg.min(axis=-1) == 0) and np.all(cg.max(axis=-1) == 3)


def test_quantizer_constant_group():
    y = np.full((1, 32), 1.2345)
    codes, scale, zero, _, _ = quant.quantize_groups(y, 32)
    assert scale[0, 0] == 0.0 and np.all(codes == 0)
    assert zero[0, 0] == quant.bf16_round(1.2345)


def test_quantizer_zero_rounded_past_the_clip():
    """A group held within a BF16 ulp of a clip that BF16 cannot represent.  R = alpha I with
    alpha = 1 + 2^-8 + 2^-10 maps 1.0 to 1.0048828125 (inside the ulp below c = 1 + 0.75 * 2^-7) and
    1.0078125 above c.  The zero rounds to 1.0078125, past the clip, and the scale is BF16 of
    2^-10 / 3 = 1.3359375 * 2^-12 (1/3 = 1.0101010...b * 2^-2 rounds up at 7 bits), so every
    (clip(y) - z) / s is at most -6: all codes are 0.  The mirrored group sits below -c: the zero
    rounds to -1.0078125 and every code is 3."""
    alpha = 1 + 2.0 ** -8 + 2.0 ** -10
    c = 1 + 0.75 * 2.0 ** -7
    row = np.repeat([1.0, 1.0078125], 16)
    x = np.concatenate([row, row, -row, -row])[None, None, :]
    q = cache.quantize_rows(x, alpha * np.eye(128), c, 32)
    s_hand = 1.3359375 * 2.0 ** -12
    assert np.array_equal(q["zero"][0, 0], [1.0078125, 1.0078125, -1.0078125, -1.0078125])
    assert np.array_equal(q["scale"][0, 0], [s_hand] * 4)
    assert np.all(q["codes"][0, 0, :64] == 0) and np.all(q["codes"][0, 0, 64:] == 3)
    # the image of the clip under (y - z) / s is about -6, not within [0, 3]
    assert (c - 1.0078125) / s_hand < -5.5


def test_quantize_with_matches_quantize_groups():
    rng = np.random.default_rng(14)
    y = rng.standard_normal((50, 128))
    codes, scale, zero, _, _ = quant.quantize_groups(y, 32)
    assert np.array_equal(quant.quantize_with(y, scale, zero, 32), codes)


# ---------------------------------------------------------------- code layouts
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("which", ["k", "v"])
def test_layout_is_bijection_and_round_trips(d, which):
    offs = quant.k_bit_offsets(d) if which == "k" else quant.v_bit_offsets(d)
    assert sorted(offs.tolist()) == list(range(0, 2 * d, 2))
    rng = np.random.default_rng(15)
    codes = rng.integers(0, 4, size=(7, 3, d)).astype(np.uint8)
    assert np.array_equal(quant.unpack_rows(quant.pack_rows(codes, offs), offs), codes)


def test_layout_hand_examples():
    # K row, d=64 (one word per lane tig): c = 32g + 16kt + 8h + 2tig at bits 2x, c+1 at 16+2x, P = 4g+2kt+h = x
    k64 = quant.k_bit_offsets(64)
    assert k64[0] == 0 and k64[1] == 16          # tig 0, slot 0
    assert k64[2] == 32 and k64[3] == 48         # tig 1 -> word 1
    assert k64[8] == 2 and k64[16] == 4          # h=1 -> slot 1; kt=1 -> slot 2
    assert k64[32] == 8 and k64[62] == 3 * 32 + 14  # g=1 -> slot 4; c=62: tig 3, slot 7
    # K row, d=128 (two words per lane): group 2 starts the second word of each lane
    k128 = quant.k_bit_offsets(128)
    assert k128[64] == 32 and k128[66] == 3 * 32  # c=66: g=2 -> P=8 -> w=1, x=0; tig 1 -> word 2*1+1
    # V row: channel 64*(hw mod (d/64)) + 8s + hw div (d/64) at bit 16*hw + 2s
    v64 = quant.v_bit_offsets(64)
    assert v64[0] == 0 and v64[1] == 16 and v64[8] == 2 and v64[63] == 16 * 7 + 14
    v128 = quant.v_bit_offsets(128)
    assert v128[0] == 0 and v128[64] == 16 and v128[1] == 32 and v128[8] == 2 and v128[127] == 16 * 15 + 14


# ---------------------------------------------------------------- attention
def _brute_attention(q, k, v):
    d = len(q)
    logits = [sum(q[c] * k[j][c] for c in range(d)) / math.sqrt(d) for j in range(len(k))]
    mx = max(logits)
    e = [math.exp(x - mx) for x in logits]
    z = sum(e)
    return np.array([sum(e[j] / z * v[j][c] for j in range(len(k))) for c in range(d)])


def test_softmax_attention_brute_force():
    rng = np.random.default_rng(16)
    q = rng.standard_normal(8)
    k = rng.standard_normal((5, 8))
    v = rng.standard_normal((5, 8))
    assert np.allclose(attention.softmax_attention(q, k, v), _brute_attention(q, k, v), rtol=1e-13, atol=1e-14)


def test_softmax_attention_special_cases():
    rng = np.random.default_rng(17)
    v = rng.standard_normal((6, 4))
    k = rng.standard_normal((6, 4))
    assert np.allclose(attention.softmax_attention(np.zeros(4), k, v), v.mean(axis=0), rtol=1e-14, atol=1e-15)
    assert np.allclose(attention.softmax_attention(rng.standard_normal(4), k[:1], v[:1]), v[0], rtol=0, atol=1e-15)


def test_dot_product_invariant_under_shared_rotation():
    wl = syn.tiny()
    q = syn.queries(wl, 0, 16, calib=True)
    k, v = syn.kv_tokens(wl, 0, 16, calib=True)
    r = rotation.layer_fixture(q, k, v)["R_K64"]
    a = syn.queries(wl, 0, 4)[:, 0, :].astype(np.float64)
    b = syn.kv_tokens(wl, 0, 4)[0][:, 0, :].astype(np.float64)
    assert np.abs((a @ r) @ (b @ r).T - a @ b.T).max() < 1e-9 * np.abs(a @ b.T).max()


def _geom(num_pages=40, d=64, p=16, s=4, w=8, hkv=2, reqs=4, layers=1):
    return cache.Geometry(layers, hkv, d, p, 32, s, w, num_pages, reqs)


def _fixture(d=64, hq=4, hkv=2, seed=21):
    wl = syn.Workload("pin", syn.Shape(hq, hkv, d, 16, 32, 4, 8, 1), [0], seed=seed, dtype="bf16")
    q = syn.queries(wl, 0, 32, calib=True)
    k, v = syn.kv_tokens(wl, 0, 32, calib=True)
    return wl, rotation.layer_fixture(q, k, v)


def _prefill(img, wl, fx, n, bt, slot=0, sub=0, layer=0):
    k, v = syn.kv_tokens(wl, layer, n, sub=sub)
    cache.write_kv(img, layer, k, v, [0, n], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"],
                   bt, [slot])
    return k, v


def test_decode_no_history_equals_brute_force():
    g = _geom()
    wl, fx = _fixture()
    img = cache.CacheImage(g)
    bt = np.arange(40, dtype=np.int32)[None, :]
    n = 10  # <= S + W: no history
    k, v = _prefill(img, wl, fx, n, bt)
    q = syn.queries(wl, 0, 1)
    out = attention.decode(img, 0, q, bt, [n], [0], fx["R_K"], fx["R_V"])
    kb = quant.bf16_round(k.astype(np.float64))
    vb = quant.bf16_round(v.astype(np.float64))
    for h in range(4):
        want = _brute_attention(q[0, h], kb[:, h // 2], vb[:, h // 2])
        assert np.allclose(out[0, h], want, rtol=1e-12, atol=1e-13)


def test_decode_with_history_brute_force_loops():
    """Mixed cache end to end against loops over the quantiser's own outputs (no packing involved)."""
    g = _geom()
    wl, fx = _fixture()
    img = cache.CacheImage(g)
    bt = np.arange(40, dtype=np.int32)[None, :]
    n = 45
    k, v = syn.kv_tokens(wl, 0, n)
    diag = cache.write_kv(img, 0, k, v, [0, n], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, [0])
    assert list(diag["t"]) == list(range(4, n - 8))
    q = syn.queries(wl, 0, 1)
    out = attention.decode(img, 0, q, bt, [n], [0], fx["R_K"], fx["R_V"])
    rk = fx["R_K"].astype(np.float64)
    rv = fx["R_V"].astype(np.float64)
    d = 64
    for h in range(4):
        kv = h // 2
        keys, vals = [], []
        for t in range(n):
            if 4 <= t < n - 8:
                m = t - 4
                for qd, dst, r in ((diag["k"], keys, rk), (diag["v"], vals, rv)):
                    yhat = [qd["zero"][m, kv, j // 32] + int(qd["codes"][m, kv, j]) * qd["scale"][m, kv, j // 32]
                            for j in range(d)]
                    dst.append([sum(yhat[i] * r[c, i] for i in range(d)) for c in range(d)])  # y_hat R^T
            else:
                keys.append(quant.bf16_round(float(k[t, kv, c])) for c in range(d))
                keys[-1] = list(keys[-1])
                vals.append([quant.bf16_round(float(v[t, kv, c])) for c in range(d)])
        want = _brute_attention(q[0, h].astype(np.float64), keys, vals)
        assert np.allclose(out[0, h], want, rtol=1e-10, atol=1e-11)


def test_decode_fused_equals_plain():
    g = _geom(d=128, p=16, s=4, w=8, hkv=2, num_pages=30)
    wl, fx = _fixture(d=128, hq=8, hkv=2)
    img = cache.CacheImage(g)
    bt = np.array([np.arange(30)], dtype=np.int32)
    n = 300
    _prefill(img, wl, fx, n, bt)
    for scale in (1.0, 0.25):
        q = syn.queries(wl, 0, 1, scale=scale)
        a = attention.decode(img, 0, q, bt, [n], [0], fx["R_K"], fx["R_V"])
        b = attention.decode_fused(img, 0, q, bt, [n], [0], fx["R_K"], fx["R_V"])
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(a).max())


# ---------------------------------------------------------------- cache logic
def test_append_chain_equals_direct_prefill():
    g = _geom()
    wl, fx = _fixture()
    bt = np.arange(40, dtype=np.int32)[None, :]
    n0, extra = 30, 9
    k, v = syn.kv_tokens(wl, 0, n0 + extra)
    a = cache.CacheImage(g)
    cache.write_kv(a, 0, k[:n0], v[:n0], [0, n0], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, [0])
    for i in range(extra):
        cache.append_step(a, 0, k[n0 + i][None], v[n0 + i][None], [n0 + i], fx["R_K"], fx["R_V"],
                          fx["clip_K"], fx["clip_V"], bt, [0])
    b = cache.CacheImage(g)
    cache.write_kv(b, 0, k, v, [0, n0 + extra], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, [0])
    assert np.array_equal(a.pool, b.pool)
    assert np.array_equal(a.slab, b.slab)


def test_eviction_moves_oldest_recent_token():
    g = _geom()
    wl, fx = _fixture()
    bt = np.arange(40, dtype=np.int32)[None, :]
    n0 = 20
    k, v = syn.kv_tokens(wl, 0, n0 + 1)
    img = cache.CacheImage(g)
    cache.write_kv(img, 0, k[:n0], v[:n0], [0, n0], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, [0])
    e = n0 - 8
    diag = cache.append_step(img, 0, k[n0][None], v[n0][None], [n0], fx["R_K"], fx["R_V"], fx["clip_K"],
                             fx["clip_V"], bt, [0])
    assert list(diag["t"]) == [e]
    assert cache.window_slot(e, 4, 8) == cache.window_slot(n0, 4, 8)
    kw, _ = img.read_window(0, 0, n0)
    assert np.array_equal(kw, quant.bf16_round(k[n0].astype(np.float64)))


def test_decode_invariant_under_block_table_permutation():
    g = _geom()
    wl, fx = _fixture()
    n = 200
    q = syn.queries(wl, 0, 1)
    outs = []
    for order in (np.arange(40), syn.page_permutation(3, 40)):
        img = cache.CacheImage(g, fill=0xFF)
        bt = np.asarray(order, dtype=np.int32)[None, :]
        _prefill(img, wl, fx, n, bt)
        outs.append(attention.decode(img, 0, q, bt, [n], [0], fx["R_K"], fx["R_V"]))
    assert np.array_equal(outs[0], outs[1])


def test_shared_prefix_equals_materialised_copy():
    """Fork at a branch point (shared full pages, copied partial page and window) then diverge."""
    g = _geom(num_pages=64)
    wl, fx = _fixture()
    n_pre, n = 64, 150  # history of the prefix = [4, 56): pages 0-2 full, page 3 partial
    k, v = syn.kv_tokens(wl, 0, n)
    k2, v2 = syn.kv_tokens(wl, 0, n, sub=1)
    k2[:n_pre], v2[:n_pre] = k[:n_pre], v[:n_pre]
    args = (fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"])
    sh = cache.CacheImage(g)
    bt = np.full((2, 20), -1, dtype=np.int32)
    bt[0, :10] = np.arange(10)
    bt[1, :3] = np.arange(3)            # shared full pages
    bt[1, 3:10] = np.arange(10, 17)     # page 3 copied to 10, rest private
    cache.write_kv(sh, 0, k[:n_pre], v[:n_pre], [0, n_pre], [0], *args, bt[:1], [0])
    cache.fork_prefix(sh, 0, 1, bt[0], bt[1], n_pre)
    cache.write_kv(sh, 0, k[n_pre:], v[n_pre:], [0, n - n_pre], [n_pre], *args, bt[:1], [0])
    cache.write_kv(sh, 0, k2[n_pre:], v2[n_pre:], [0, n - n_pre], [n_pre], *args, bt[1:], [1])
    mat = cache.CacheImage(g)
    bt2 = bt.copy()
    bt2[1, :10] = np.arange(20, 30)
    cache.write_kv(mat, 0, k, v, [0, n], [0], *args, bt2[:1], [0])
    cache.write_kv(mat, 0, k2, v2, [0, n], [0], *args, bt2[1:], [1])
    q = syn.queries(wl, 0, 2)
    a = attention.decode(sh, 0, q, bt, [n, n], [0, 1], fx["R_K"], fx["R_V"])
    b = attention.decode(mat, 0, q, bt2, [n, n], [0, 1], fx["R_K"], fx["R_V"])
    assert np.array_equal(a, b)
    with pytest.raises(ValueError):
        bad = bt[1].copy()
        bad[0] = 40
        cache.fork_prefix(sh, 0, 1, bt[0], bad, n_pre)


def test_bf16_paged_decode_matches_textbook():
    rng = np.random.default_rng(22)
    hkv, p, d, n = 2, 4, 8, 11
    k = quant.bf16_round(rng.standard_normal((n, hkv, d)))
    v = quant.bf16_round(rng.standard_normal((n, hkv, d)))
    pool = np.zeros((1, 6, hkv, 2, p, d), dtype=np.uint16)
    bt = np.array([[5, 2, 0]], dtype=np.int32)
    for t in range(n):
        pool[0, bt[0, t // p], :, 0, t % p] = quant.bf16_to_bits(k[t])
        pool[0, bt[0, t // p], :, 1, t % p] = quant.bf16_to_bits(v[t])
    q = rng.standard_normal((1, 4, d))
    out = attention.bf16_paged_decode(pool, 0, q, bt, [n], p)
    for h in range(4):
        assert np.allclose(out[0, h], _brute_attention(q[0, h], k[:, h // 2], v[:, h // 2]), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- extend (chunked prefill) attention
def _sdpa(q, k, v, mask):
    """torch's scaled_dot_product_attention in float64 on the CPU: q [T, Hq, d], k, v [N, Hkv, d],
    mask [T, N] (True = visible); kv heads repeated to the query heads."""
    import torch
    grp = q.shape[1] // k.shape[1]
    tq = torch.from_numpy(np.asarray(q, np.float64)).permute(1, 0, 2)
    tk = torch.from_numpy(np.asarray(k, np.float64)).permute(1, 0, 2).repeat_interleave(grp, dim=0)
    tv = torch.from_numpy(np.asarray(v, np.float64)).permute(1, 0, 2).repeat_interleave(grp, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(mask))
    return out.permute(1, 0, 2).numpy()


def _chunk(wl, n, sub=1):
    k, v = syn.kv_tokens(wl, 0, n, sub=sub)
    return quant.bf16_round(k.astype(np.float64)), quant.bf16_round(v.astype(np.float64))


def test_extend_without_prefix_is_causal_sdpa():
    g = _geom()
    wl, fx = _fixture()
    img = cache.CacheImage(g)
    bt = np.arange(40, dtype=np.int32)[None, :]
    t = 23
    k, v = _chunk(wl, t)
    q = syn.queries(wl, 0, t, sub=3)
    out = attention.extend(img, 0, q, k, v, [0, t], [0], bt, [0], fx["R_K"], fx["R_V"])
    want = _sdpa(q, k, v, np.tril(np.ones((t, t), dtype=bool)))
    assert np.allclose(out, want, rtol=1e-12, atol=1e-13)


def test_extend_over_a_bf16_prefix_is_masked_sdpa():
    """Prefix short enough to be all sink + recent (no INT2 history): keys = BF16 prefix ++ chunk."""
    g = _geom()
    wl, fx = _fixture()
    img = cache.CacheImage(g)
    bt = np.arange(40, dtype=np.int32)[None, :]
    n_pre, t = 11, 9    # 11 <= S + W = 12
    kp, vp = _prefill(img, wl, fx, n_pre, bt)
    k, v = _chunk(wl, t)
    q = syn.queries(wl, 0, t, sub=3)
    out = attention.extend(img, 0, q, k, v, [0, t], [n_pre], bt, [0], fx["R_K"], fx["R_V"])
    keys = np.concatenate([quant.bf16_round(kp.astype(np.float64)), k])
    vals = np.concatenate([quant.bf16_round(vp.astype(np.float64)), v])
    mask = np.concatenate([np.ones((t, n_pre), dtype=bool), np.tril(np.ones((t, t), dtype=bool))], axis=1)
    assert np.allclose(out, _sdpa(q, keys, vals, mask), rtol=1e-12, atol=1e-13)


def test_extend_with_an_invisible_chunk_token_is_decode_over_the_prefix():
    """A one-token chunk whose key scores -1e6 * |q|^2 has weight exactly 0 in float64, so extend
    reduces to decode over the cached prefix (INT2 history, rotated back, plus the BF16 window)."""
    g = _geom(hkv=2)
    wl, fx = _fixture()
    img = cache.CacheImage(g)
    bt = np.arange(40, dtype=np.int32)[None, :]
    n_pre = 45   # history tokens 4 .. 36
    _prefill(img, wl, fx, n_pre, bt)
    q = syn.queries(wl, 0, 1, sub=3).astype(np.float64)
    q[0, 1] = q[0, 0]   # both query heads of kv head 0 alike, and of kv head 1
    q[0, 3] = q[0, 2]
    k = np.stack([-1e6 * q[0, 0], -1e6 * q[0, 2]])[None]
    v = np.full_like(k, 7.0)
    out = attention.extend(img, 0, q, k, v, [0, 1], [n_pre], bt, [0], fx["R_K"], fx["R_V"])
    want = attention.decode(img, 0, q, bt, [n_pre], [0], fx["R_K"], fx["R_V"])
    assert np.array_equal(out, want)


def test_extend_is_causal_and_requests_are_independent():
    g = _geom()
    wl, fx = _fixture()
    img = cache.CacheImage(g)
    bt = np.arange(40, dtype=np.int32).reshape(2, 20)
    lens_pre, lens = [37, 5], [6, 4]
    _prefill(img, wl, fx, lens_pre[0], bt, slot=0, sub=0)
    cache.write_kv(img, 0, *syn.kv_tokens(wl, 0, lens_pre[1], sub=5), [0, lens_pre[1]], [0], fx["R_K"], fx["R_V"],
                   fx["clip_K"], fx["clip_V"], bt[1:], [1])
    k, v = _chunk(wl, sum(lens))
    q = syn.queries(wl, 0, sum(lens), sub=3)
    cu = [0, lens[0], sum(lens)]
    both = attention.extend(img, 0, q, k, v, cu, lens_pre, bt, [0, 1], fx["R_K"], fx["R_V"])
    # request 1 alone (its own block-table row and slot)
    alone = attention.extend(img, 0, q[lens[0]:], k[lens[0]:], v[lens[0]:], [0, lens[1]], lens_pre[1:], bt[1:], [1],
                             fx["R_K"], fx["R_V"])
    assert np.array_equal(both[lens[0]:], alone)
    # changing chunk token j changes no output before j
    k2, v2 = k.copy(), v.copy()
    k2[3] += 5.0
    v2[3] -= 5.0
    moved = attention.extend(img, 0, q, k2, v2, cu, lens_pre, bt, [0, 1], fx["R_K"], fx["R_V"])
    assert np.array_equal(moved[:3], both[:3])
    assert not np.allclose(moved[3:lens[0]], both[3:lens[0]])
    assert np.array_equal(moved[lens[0]:], both[lens[0]:])


def test_extend_is_invariant_under_within_group_channel_permutation():
    """R' = R P with P permuting channels inside each group of 32: every group keeps its values (same
    min, max, scale, zero), the codes move with the channels, and y_hat' R'^T = y_hat R^T.  So extend
    over a prefix written with R' equals extend over the prefix written with R (history, window and
    chunk all visible); a transposed or misapplied R in the rotate-back breaks the equality."""
    g = _geom(num_pages=40, d=64, p=16, s=4, w=8, hkv=2)
    wl, fx = _fixture()
    rng = np.random.default_rng(5)
    perm = np.concatenate([32 * gi + rng.permutation(32) for gi in range(2)])
    outs = []
    for rk, rv in ((fx["R_K"], fx["R_V"]), (fx["R_K"][:, perm], fx["R_V"][:, perm])):
        img = cache.CacheImage(g)
        bt = np.arange(40, dtype=np.int32)[None, :]
        k, v = syn.kv_tokens(wl, 0, 90)
        cache.write_kv(img, 0, k, v, [0, 90], [0], rk, rv, fx["clip_K"], fx["clip_V"], bt, [0])
        kc, vc = _chunk(wl, 6)
        q = syn.queries(wl, 0, 6, sub=3)
        outs.append(attention.extend(img, 0, q, kc, vc, [0, 6], [90], bt, [0], rk, rv))
    assert np.allclose(outs[0], outs[1], rtol=1e-12, atol=1e-12)
    assert not np.allclose(outs[0], 0.0)


# ---------------------------------------------------------------- per-kv-head rotations
def _head_fixture(d=64, hq=4, hkv=2, seed=23):
    wl = syn.Workload("pinh", syn.Shape(hq, hkv, d, 16, 32, 4, 8, 1), [0], seed=seed, dtype="bf16")
    q = syn.queries(wl, 0, 32, calib=True)
    k, v = syn.kv_tokens(wl, 0, 32, calib=True)
    return wl, rotation.head_fixture(q, k, v)


def test_head_fixture_rotations_orthogonal_and_distinct():
    _, fx = _head_fixture()
    for key in ("R_K64", "R_V64"):
        r = fx[key]
        assert r.shape == (2, 64, 64)
        for h in range(2):
            assert np.abs(r[h] @ r[h].T - np.eye(64)).max() < 1e-12
        assert np.abs(r[0] - r[1]).max() > 1e-3  # each kv head is calibrated on its own data


def test_per_head_rotation_is_each_heads_own_rotation():
    """Head h of a per-head quantisation equals quantising head h alone with its rotation (catches a
    head / rotation mix-up or a transposed rotation)."""
    wl, fx = _head_fixture()
    x, _ = syn.kv_tokens(wl, 0, 50)
    got = cache.quantize_rows(x, fx["R_K"], fx["clip_K"], 32)
    for h in range(2):
        one = cache.quantize_rows(x[:, h:h + 1], fx["R_K"][h], fx["clip_K"], 32)
        for key in ("y", "codes", "scale", "zero"):
            assert np.array_equal(got[key][:, h:h + 1], one[key])
    # a transposed rotation gives other values
    bad = cache.quantize_rows(x, np.transpose(fx["R_K"], (0, 2, 1)), fx["clip_K"], 32)
    assert not np.array_equal(bad["codes"], got["codes"])


def test_per_head_rotations_all_equal_reproduce_the_shared_rotation():
    """Per-kv-head rotations that are all the layer's rotation give the shared path's codes, scales and
    zeros bit for bit, and its decode output."""
    g = _geom()
    wl, fx = _fixture()
    stack = lambda r: np.stack([r, r])
    x, _ = syn.kv_tokens(wl, 0, 60)
    a = cache.quantize_rows(x, fx["R_K"], fx["clip_K"], 32)
    b = cache.quantize_rows(x, stack(fx["R_K"]), fx["clip_K"], 32)
    for key in ("codes", "scale", "zero"):
        assert np.array_equal(a[key], b[key])
    assert np.abs(a["y"] - b["y"]).max() <= 1e-14 * np.abs(a["y"]).max()
    bt = np.arange(40, dtype=np.int32)[None, :]
    img1, img2 = cache.CacheImage(g), cache.CacheImage(g)
    n = 200
    k, v = syn.kv_tokens(wl, 0, n)
    cache.write_kv(img1, 0, k, v, [0, n], [0], fx["R_K"], fx["R_V"], fx["clip_K"], fx["clip_V"], bt, [0])
    cache.write_kv(img2, 0, k, v, [0, n], [0], stack(fx["R_K"]), stack(fx["R_V"]), fx["clip_K"], fx["clip_V"], bt,
                   [0])
    assert np.array_equal(img1.pool, img2.pool) and np.array_equal(img1.slab, img2.slab)
    q = syn.queries(wl, 0, 1)
    o1 = attention.decode(img1, 0, q, bt, [n], [0], fx["R_K"], fx["R_V"])
    o2 = attention.decode(img2, 0, q, bt, [n], [0], stack(fx["R_K"]), stack(fx["R_V"]))
    assert np.abs(o1 - o2).max() <= 1e-13 * np.abs(o1).max()


def test_per_head_decode_fused_equals_plain():
    """Rotating each query by its kv head's R_K and applying that head's R_V^T once is exact."""
    g = _geom(d=64, p=16, s=4, w=8, hkv=2, num_pages=30)
    wl, fx = _head_fixture()
    img = cache.CacheImage(g)
    bt = np.array([np.arange(30)], dtype=np.int32)
    n = 300
    _prefill(img, wl, fx, n, bt)
    for scale in (1.0, 0.25):
        q = syn.queries(wl, 0, 1, scale=scale)
        a = attention.decode(img, 0, q, bt, [n], [0], fx["R_K"], fx["R_V"])
        b = attention.decode_fused(img, 0, q, bt, [n], [0], fx["R_K"], fx["R_V"])
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(a).max())
        # decoding with the other head's rotations is wrong: the rotations are used per head
        swapped = attention.decode(img, 0, q, bt, [n], [0], fx["R_K"][::-1], fx["R_V"][::-1])
        assert np.abs(a - swapped).max() > 1e-3 * np.abs(a).max()
