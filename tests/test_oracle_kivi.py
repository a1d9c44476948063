"""Pins of the oracle's KIVI quantisation, packing and attention (CPU only).

What pins each part:
  * scale bits    -- numpy's float16 rounding of (max - min) / (2^b - 1), and exact
                     rational rounding with ``fractions`` (pins the fp64 -> fp16 step)
  * codes         -- brute force: the code is the grid point nearest to x, ties to even
  * error bound   -- |x - x_hat| <= scale / 2 except where the top code is clamped
  * flush rule    -- a token-by-token residual simulation equals the closed form n_q
  * packing       -- an unpacker written from the layout statement round-trips and
                     every code bit lands in exactly one place
  * attention     -- with the whole sequence in the residual (R >= T) it is full
                     attention; otherwise SDPA (fp64) over the dequantised grid values
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

G = 32


def _groups(rng, n, kind):
    if kind == "normal":
        return rng.standard_normal((n, G)).astype(np.float16)
    if kind == "offset":
        return (rng.standard_normal((n, G)) + rng.uniform(-2, 2, (n, 1))).astype(np.float16)
    if kind == "wide":
        return (rng.standard_normal((n, G)) * 10.0 ** rng.uniform(-6, 4, (n, 1))).astype(np.float16)
    if kind == "coarse":  # few distinct values -> many exact ties
        return (rng.integers(-8, 8, (n, G)) * 0.25).astype(np.float16)
    raise ValueError(kind)


def _quant_one_group_v(orc, x16, bits):
    """Use the V path (per token, one channel group of 32) to quantise one group."""
    T = G  # one V group per token row; put the values in token 0's first channel group
    D = G
    V = np.zeros((T, D), np.float16)
    V[0] = x16
    K = np.zeros((T, D), np.float16)
    r = orc.kivi_quantize_unit(K, V, G, bits)
    return r["v_scale"][0, 0], r["v_zero"][0, 0], r["v_codes"][0]


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kind", ["normal", "offset", "wide", "coarse"])
def test_scale_zero_and_codes_brute_force(orc, bits, kind):
    rng = np.random.default_rng(bits * 10 + len(kind))
    xs = _groups(rng, 64, kind)
    cmax = (1 << bits) - 1
    for x16 in xs:
        sb, zb, codes = _quant_one_group_v(orc, x16, bits)
        x = x16.astype(np.float64)
        mn, mx = x.min(), x.max()
        # zero: the group minimum (+0 for a zero minimum)
        assert np.float16(mn).view(np.uint16) == zb or (mn == 0 and zb == 0)
        # scale: binary16 RNE of the exact quotient (numpy's rounding, independent code)
        assert np.float16(np.float64(mx - mn) / cmax).view(np.uint16) == sb
        # ... and of the exact rational quotient (pins the double rounding step)
        exact = Fraction(float(mx)) - Fraction(float(mn))
        q = exact / cmax
        cands = np.array([sb - 1, sb, sb + 1], np.uint16)
        vals = [Fraction(float(c.view(np.float16))) for c in cands if c < 0x7c00]
        best = min(vals, key=lambda v: (abs(v - q), int(np.float16(float(v)).view(np.uint16)) & 1))
        assert np.float16(float(best)).view(np.uint16) == sb
        s = float(np.uint16(sb).view(np.float16))
        z = float(np.uint16(zb).view(np.float16))
        if s == 0.0:
            assert np.all(codes == 0)
            continue
        # brute force over every code: nearest grid point, ties to the even code
        grid = z + np.arange(cmax + 1, dtype=np.float64) * s      # exact in fp64
        ref = []
        for xi in x:
            dist = np.abs(xi - grid)                              # exact in fp64
            idx = np.flatnonzero(dist == dist.min())
            ref.append(idx[0] if len(idx) == 1 else [c for c in idx if c % 2 == 0][0])
        assert np.array_equal(codes, np.array(ref))
        # error bound: half a step, except where the top code is clamped
        err = np.abs(x - (z + codes * s))
        clamped = codes == cmax
        assert np.all(err[~clamped] <= s / 2)
        assert np.all(err[clamped] <= max(s / 2, (mx - mn) - cmax * s))


def test_exact_ties_go_to_even(orc):
    # values on exact half-grid points: zero = 0, max = 15 -> scale = 1, x = k + 0.5
    x = np.array([0.0, 15.0] + [k + 0.5 for k in range(15)] + [3.0] * 15, np.float16)
    sb, zb, codes = _quant_one_group_v(orc, x, 4)
    assert float(np.uint16(sb).view(np.float16)) == 1.0 and zb == 0
    half = codes[2:17]
    expect = [k if k % 2 == 0 else k + 1 for k in range(15)]
    assert list(half) == expect


def test_degenerate_and_negative_zero(orc):
    x = np.full(G, 1.5, np.float16)
    sb, zb, codes = _quant_one_group_v(orc, x, 4)
    assert sb == 0 and np.float16(1.5).view(np.uint16) == zb and np.all(codes == 0)
    x = np.array([-0.0] * 16 + [0.0] * 16, np.float16)
    sb, zb, codes = _quant_one_group_v(orc, x, 2)
    assert sb == 0 and zb == 0
    x = np.array([-0.0] + [1.0] * 31, np.float16)
    sb, zb, _ = _quant_one_group_v(orc, x, 4)
    assert zb == 0 and np.uint16(sb).view(np.float16) == np.float16(1.0 / 15)


def test_k_is_per_channel_v_is_per_token(orc):
    rng = np.random.default_rng(11)
    T, D = 64, 64
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    r = orc.kivi_quantize_unit(K, V, T, 4)
    k = K.astype(np.float64)
    for g in range(T // G):
        blk = k[g * G:(g + 1) * G]
        assert np.array_equal(r["k_zero"][g], blk.min(0).astype(np.float16).view(np.uint16))
        assert np.array_equal(r["k_scale"][g],
                              ((blk.max(0) - blk.min(0)) / 15).astype(np.float16).view(np.uint16))
    v = V.astype(np.float64).reshape(T, D // G, G)
    assert np.array_equal(r["v_zero"], v.min(2).astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("R", [0, 16, 128, 100])
def test_flush_rule_simulation(orc, R):
    """Append tokens one by one into a residual; once it holds R + G tokens the oldest G are
    quantised.  The simulated quantised count equals the closed form at every length."""
    n_q = 0
    for T in range(1, 700):
        n_res = T - n_q
        while n_res >= R + G:
            n_q += G
            n_res -= G
        assert orc.kivi_nq(T, R) == n_q
        assert 0 <= T - n_q < R + G
    assert orc.kivi_nq(4096, 128) == 3968 and orc.kivi_nq(2048, 128) == 1920


def _unpack_from_spec(kb, vb, D, bits):
    """Unpacker written from the block layout statement in include/kvc.h."""
    WK = D * bits // 32
    per_word = 32 // bits
    mask = (1 << bits) - 1
    kw = kb[:G * WK * 4].view(np.uint32).reshape(G, WK)
    kc = np.zeros((G, D), np.uint8)
    for t in range(G):
        for w in range(WK):
            for i in range(per_word):
                kc[t, per_word * w + i] = (int(kw[t, w]) >> (bits * i)) & mask
    ks = kb[G * WK * 4:].view(np.uint16)
    W = D * bits // 128
    vw = vb[:G * WK * 4].view(np.uint32).reshape(G // 2, 8, W)
    vc = np.full((G, D), 255, np.uint8)
    for i in range(G // 2):
        for r in range(8):
            for k in range(W):
                word = int(vw[i, (r + 2 * i) % 8, k])
                for j in range(16 // bits):
                    d = 16 * (k * (8 // bits) + j // 2) + 8 * (j % 2) + r
                    assert vc[2 * i, d] == 255 and vc[2 * i + 1, d] == 255
                    vc[2 * i, d] = (word >> (bits * j)) & mask
                    vc[2 * i + 1, d] = (word >> (16 + bits * j)) & mask
    vs = vb[G * WK * 4:].view(np.uint16).reshape(2, D // G, G)
    return kc, ks[:D], ks[D:], vc, vs[0].T, vs[1].T


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bits", [2, 4])
def test_pack_layout_round_trip(orc, D, bits):
    rng = np.random.default_rng(D + bits)
    K = rng.standard_normal((2 * G, D)).astype(np.float16)
    V = rng.standard_normal((2 * G, D)).astype(np.float16)
    r = orc.kivi_quantize_unit(K, V, 2 * G, bits)
    kb, vb = orc.kivi_pack_unit(r, D, bits)
    assert kb.shape == (2, orc.kivi_block_bytes(D, bits)) and kb.shape[1] % 16 == 0
    for g in range(2):
        kc, ks, kz, vc, vs, vz = _unpack_from_spec(kb[g], vb[g], D, bits)
        assert np.array_equal(kc, r["k_codes"][g * G:(g + 1) * G])
        assert np.array_equal(vc, r["v_codes"][g * G:(g + 1) * G])
        assert np.array_equal(ks, r["k_scale"][g]) and np.array_equal(kz, r["k_zero"][g])
        assert np.array_equal(vs, r["v_scale"][g * G:(g + 1) * G])
        assert np.array_equal(vz, r["v_zero"][g * G:(g + 1) * G])
    # every code bit is used: all-max codes give all-ones code words
    full = {k: (np.full_like(v, (1 << bits) - 1) if k.endswith("codes") else v) for k, v in r.items()}
    kb, vb = orc.kivi_pack_unit(full, D, bits)
    nbytes = G * D * bits // 8
    assert np.all(kb[:, :nbytes] == 255) and np.all(vb[:, :nbytes] == 255)


def test_attention_all_residual_equals_full(orc):
    rng = np.random.default_rng(5)
    T, D, g = 40, 64, 2
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    q = rng.standard_normal((g, D)).astype(np.float16)
    out, lse = orc.kivi_attend_unit(q, K, V, T, R=T, bits=4)
    ref, ref_lse, _ = orc.decode_attend(q[None], K[None, None], V[None, None],
                                        np.array([[T]], np.int32))
    assert np.array_equal(out, ref[0]) and np.array_equal(lse, ref_lse[0])


@pytest.mark.parametrize("bits", [2, 4])
def test_attention_over_dequantised_grid_matches_sdpa(orc, bits):
    rng = np.random.default_rng(50 + bits)
    T, D, g, R = 150, 128, 3, 16
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = (rng.standard_normal((T, D)) + 1.5).astype(np.float16)
    q = rng.standard_normal((g, D)).astype(np.float16)
    n_q = orc.kivi_nq(T, R)
    r = orc.kivi_quantize_unit(K[:n_q], V[:n_q], n_q, bits)
    # dequantised grid values: zero + code * scale (every value checked nearest by brute force)
    ks = r["k_scale"].view(np.float16).astype(np.float64).repeat(G, 0)
    kz = r["k_zero"].view(np.float16).astype(np.float64).repeat(G, 0)
    vs = r["v_scale"].view(np.float16).astype(np.float64).repeat(G, 1)
    vz = r["v_zero"].view(np.float16).astype(np.float64).repeat(G, 1)
    Kh = np.concatenate([kz + r["k_codes"] * ks, K[n_q:].astype(np.float64)])
    Vh = np.concatenate([vz + r["v_codes"] * vs, V[n_q:].astype(np.float64)])
    out, _ = orc.kivi_attend_unit(q, K, V, T, R=R, bits=bits, qz=r)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.astype(np.float64))[None, :, None], torch.from_numpy(Kh)[None, None],
        torch.from_numpy(Vh)[None, None])[0, :, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
