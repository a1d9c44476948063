"""Pins of the GEAR-4 oracle (oracle/gear.py) against what the definition and mathematics fix:
a group on the 4-bit grid has no residual; the sparse part holds the largest residuals; the
rank-2 factors satisfy the optimality conditions of the truncated SVD; with no sparse part and
rank 0 the attention is KIVI's (the independent C oracle); the attention is SDPA over the
reconstruction."""
import numpy as np
import pytest
import torch

from oracle import gear as gr

G = 32


def test_side_block_size():
    assert gr.n_sparse(128) == 82 and gr.n_sparse(64) == 41      # ceil(2% of 32 x D)
    assert gr.side_bytes(128) == 976 and gr.side_bytes(64) == 560


def _grid_group(rng, D):
    """Values exactly on a 4-bit grid: zero -1, scale 1/16, codes with 0 and 15 present in every
    K channel and every V (token, 32-channel group): code 0 where (t + d) % 32 == 0, 15 where it
    is 1, random elsewhere."""
    c = rng.integers(0, 16, (G, D))
    td = (np.arange(G)[:, None] + np.arange(D)[None, :]) % 32
    c[td == 0], c[td == 1] = 0, 15
    x = (-1.0 + c / 16.0).astype(np.float16)
    assert np.array_equal(x.astype(np.float64), -1.0 + c / 16.0)   # exactly representable
    return x, c


@pytest.mark.parametrize("D", [128, 64])
def test_grid_valued_group_has_no_residual(orc, D):
    rng = np.random.default_rng(D)
    X, c = _grid_group(rng, D)
    gz = gr.quantize_unit(X, X, G, 4)
    assert np.array_equal(gz["qz"]["k_codes"], c) and np.array_equal(gz["qz"]["v_codes"], c)
    for p in (gz["k"][0], gz["v"][0]):
        assert not p["E"].any() and not p["val"].astype(np.float64).any()
        np.testing.assert_array_equal(gr.reconstruct(p), X.astype(np.float64))


@pytest.mark.parametrize("seed", range(4))
def test_sparse_part_holds_the_largest_residuals(orc, seed):
    rng = np.random.default_rng(seed)
    D = 128
    K = (rng.standard_normal((G, D)) * rng.uniform(0.1, 3, (1, D))).astype(np.float16)
    V = np.round(rng.standard_normal((G, D)) * 4).astype(np.float16) / 4   # many equal residuals
    gz = gr.quantize_unit(K, V.astype(np.float16), G, 4)
    for p in (gz["k"][0], gz["v"][0]):
        a = np.abs(p["E"].astype(np.float64)).reshape(-1)
        sel = np.zeros(a.size, bool)
        sel[p["idx"].astype(np.int64)] = True
        assert sel.sum() == gr.n_sparse(D) and np.all(np.diff(p["idx"].astype(np.int64)) > 0)
        lo = a[sel].min()
        assert np.all(a[~sel] <= lo)
        # at the threshold the lower flat indices win
        tied_out = np.flatnonzero(~sel & (a == lo))
        tied_in = np.flatnonzero(sel & (a == lo))
        if tied_out.size and tied_in.size:
            assert tied_in.max() < tied_out.min()
        np.testing.assert_array_equal(p["val"], p["E"].reshape(-1)[sel].astype(np.float16))


@pytest.mark.parametrize("seed", range(4))
def test_rank2_factors_are_the_truncated_svd(orc, seed):
    """A has orthonormal rows; the residual R - L is orthogonal to the captured right subspace
    ((R - L) B^T = 0, true only for singular subspaces); |R - L|^2 = |R|^2 - |B|^2 with |B|^2
    the two largest eigenvalues of R R^T (eigvalsh, another routine); no random rank-2
    projection of R does better."""
    rng = np.random.default_rng(100 + seed)
    D = 128
    K = rng.standard_normal((G, D)).astype(np.float16)
    p = gr.quantize_unit(K, K, G, 4)["k"][0]
    R, A, B = p["R"], p["A"], p["B"]
    np.testing.assert_allclose(A @ A.T, np.eye(2), atol=1e-12)
    Lr = A.T @ B
    np.testing.assert_allclose((R - Lr) @ B.T, 0, atol=1e-10 * np.abs(R).max() ** 2 * D)
    ev = np.linalg.eigvalsh(R @ R.T)
    err = np.sum((R - Lr) ** 2)
    assert err == pytest.approx(np.sum(R ** 2) - np.sum(B ** 2), rel=1e-10)
    assert np.sum(B ** 2) == pytest.approx(ev[-1] + ev[-2], rel=1e-10)
    for _ in range(50):
        Q, _ = np.linalg.qr(rng.standard_normal((G, 2)))
        assert err <= np.sum((R - Q @ Q.T @ R) ** 2) + 1e-12


def test_no_sparse_no_rank_is_kivi(orc):
    """pct 0 and rank 0 leave only the quantised values (rounded once to fp32): the attention
    matches the C oracle's KIVI attention within that rounding."""
    rng = np.random.default_rng(7)
    T, R, D, g = 200, 40, 128, 4
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    q = rng.standard_normal((g, D)).astype(np.float16)
    o_g, l_g = gr.attend_unit(q, K, V, T, R, 4, pct=0, rank=0)
    o_k, l_k = orc.kivi_attend_unit(q, K, V, T, R, 4)
    np.testing.assert_allclose(o_g, o_k, atol=1e-6)
    np.testing.assert_allclose(l_g, l_k, atol=1e-6)


def test_attention_is_sdpa_over_the_reconstruction(orc):
    rng = np.random.default_rng(8)
    T, R, D, g = 170, 32, 64, 3
    K = rng.standard_normal((T, D)).astype(np.float16)
    V = rng.standard_normal((T, D)).astype(np.float16)
    q = rng.standard_normal((g, D)).astype(np.float16)
    n_q = orc.kivi_nq(T, R)
    gz = gr.quantize_unit(K[:n_q], V[:n_q], n_q, 4)
    o, _ = gr.attend_unit(q, K, V, T, R, 4, gz=gz)
    Kh = np.concatenate([gr.reconstruct(p) for p in gz["k"]] + [K[n_q:].astype(np.float64)])
    Vh = np.concatenate([gr.reconstruct(p) for p in gz["v"]] + [V[n_q:].astype(np.float64)])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.astype(np.float64))[None], torch.from_numpy(Kh)[None],
        torch.from_numpy(Vh)[None])[0].numpy()
    np.testing.assert_allclose(o, ref, atol=1e-12)


def test_gear_reconstruction_is_closer_than_kivi(orc):
    rng = np.random.default_rng(9)
    D = 128
    K = (rng.standard_normal((G, D)) + rng.standard_normal((G, 1)) * rng.standard_normal((1, D))
         ).astype(np.float16)
    p = gr.quantize_unit(K, K, G, 4)["k"][0]
    x = K.astype(np.float64)
    e_kivi = np.sum((x - p["xq"].astype(np.float64)) ** 2)
    e_gear = np.sum((x - gr.reconstruct(p)) ** 2)
    assert e_gear < 0.8 * e_kivi
