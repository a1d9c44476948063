"""Pins of the oracle's binary16 conversions and its attention (CPU only).

binary16: checked exhaustively / on adversarial values against numpy's own
float16 conversions (an independent library routine).
Attention: checked against torch's scaled_dot_product_attention in fp64 on the
CPU (library routine), plus special cases with closed forms.
"""
import math

import numpy as np
import pytest
import torch


def test_half_to_double_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros are kept
    assert math.copysign(1.0, got[0x8000]) == -1.0


def test_double_to_half_matches_numpy(orc):
    rng = np.random.default_rng(7)
    xs = [rng.standard_normal(200000) * s for s in (1e-6, 1e-3, 1.0, 1e2, 3e4)]
    # every midpoint between adjacent finite binary16 values (ties), +/- a hair
    h = np.arange(0, 0x7bff, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2
    xs += [mids, -mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf)]
    xs.append(np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0**-25,
                        2.0**-25 * 1.0000001, 2.0**-24 * 1.5, 2.0**-14, 2.0**-14 * (1 - 2.0**-11)]))
    x = np.concatenate(xs)
    got = orc.double_to_half(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def _rand_case(rng, B, Hq, Hkv, C, D):
    f = lambda *s: rng.standard_normal(s).astype(np.float16)
    q, K, V = f(B, Hq, D), f(B, Hkv, C, D), f(B, Hkv, C, D)
    n = rng.integers(1, C + 1, size=(B, Hkv)).astype(np.int32)
    return q, K, V, n


@pytest.mark.parametrize("B,Hq,Hkv,C,D", [(2, 4, 4, 37, 64), (3, 8, 2, 50, 128), (1, 16, 2, 7, 64),
                                          (2, 8, 1, 33, 128)])
def test_attention_matches_torch_sdpa_fp64(orc, B, Hq, Hkv, C, D):
    rng = np.random.default_rng(B * 100 + Hq + C)
    q, K, V, n = _rand_case(rng, B, Hq, Hkv, C, D)
    out, lse, logits = orc.decode_attend(q, K, V, n, want_logits=True)
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            nn = n[b, hk]
            qt = torch.from_numpy(q[b, h].astype(np.float64))[None, None, None]
            kt = torch.from_numpy(K[b, hk, :nn].astype(np.float64))[None, None]
            vt = torch.from_numpy(V[b, hk, :nn].astype(np.float64))[None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, 0, 0].numpy()
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-12)
            lg = logits[b, h, :nn]
            ref_lse = torch.logsumexp(torch.from_numpy(lg), 0).item()
            assert abs(lse[b, h] - ref_lse) < 1e-12
            ref_lg = (kt[0, 0] @ qt[0, 0, 0]).numpy() / math.sqrt(D)
            np.testing.assert_allclose(lg, ref_lg, rtol=1e-13, atol=1e-13)


def test_attention_special_cases(orc):
    rng = np.random.default_rng(3)
    B, H, C, D = 1, 2, 9, 64
    q, K, V, _ = _rand_case(rng, B, H, H, C, D)
    # one slot -> the output is that slot's value exactly
    out, lse, _ = orc.decode_attend(q, K, V, np.ones((B, H), np.int32))
    assert np.array_equal(out[0, 0], V[0, 0, 0].astype(np.float64))
    # constant values -> output equals the constant (probabilities sum to one)
    Vc = np.broadcast_to(V[:, :, :1], V.shape).copy()
    out, _, _ = orc.decode_attend(q, K, Vc, np.full((B, H), C, np.int32))
    np.testing.assert_allclose(out[0, 1], Vc[0, 1, 0].astype(np.float64), rtol=0, atol=1e-14)
    # identical keys -> uniform weights -> mean of the values
    Ks = np.broadcast_to(K[:, :, :1], K.shape).copy()
    out, lse, _ = orc.decode_attend(q, Ks, V, np.full((B, H), C, np.int32))
    np.testing.assert_allclose(out[0, 0], V[0, 0].astype(np.float64).mean(0), atol=1e-14)
    logit = float(q[0, 0].astype(np.float64) @ Ks[0, 0, 0].astype(np.float64)) / 8.0
    assert abs(lse[0, 0] - (logit + math.log(C))) < 1e-12
    # empty cache -> zero output, -inf log-sum-exp
    out, lse, _ = orc.decode_attend(q, K, V, np.zeros((B, H), np.int32))
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_gqa_head_mapping_is_contiguous(orc):
    """Query head h must read KV head h // g: make KV heads distinguishable by their values."""
    B, Hq, Hkv, C, D = 1, 8, 2, 5, 64
    q = np.zeros((B, Hq, D), np.float16)
    K = np.zeros((B, Hkv, C, D), np.float16)
    V = np.zeros((B, Hkv, C, D), np.float16)
    V[0, 0] = 1.0
    V[0, 1] = -2.0
    out, _, _ = orc.decode_attend(q, K, V, np.full((B, Hkv), C, np.int32))
    assert np.all(out[0, :4] == 1.0) and np.all(out[0, 4:] == -2.0)
