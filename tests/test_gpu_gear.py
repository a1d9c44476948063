"""GEAR-4 on the GPU against the oracle (oracle/gear.py): the KIVI blocks and the sparse parts
(indices and binary16 values) are bit-exact; the rank-2 factors, which the GPU finds by subspace
iteration rather than an SVD, must be orthonormal and reach the optimal truncation error of the
oracle's SVD within a stated margin; decode attention over the reconstruction matches the
oracle's."""
import numpy as np
import pytest
import torch

from helpers import assert_o_close, device_status_clean, np16
from oracle import gear as gr
from oracle import kivi_nq, kivi_pack_unit

pytestmark = pytest.mark.gpu
G = 32


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def _side_parts(block, D):
    """Decode one side block: (flat indices, values, A [2, 32], B [2, D])."""
    ns = gr.n_sparse(D)
    b = np.asarray(block, np.uint8)
    idx = b[:2 * ns].view(np.uint16).astype(np.int64)
    val = b[2 * ns:4 * ns].view(np.float16)
    A = b[4 * ns:4 * ns + 4 * G].view(np.float16).astype(np.float64).reshape(2, G)
    B = b[4 * ns + 4 * G:4 * ns + 4 * G + 4 * D].view(np.float16).astype(np.float64).reshape(2, D)
    return idx, val, A, B


def _check_group(gpu_side, ref, D):
    idx, val, A, B = _side_parts(gpu_side, D)
    assert np.array_equal(idx, ref["idx"].astype(np.int64))
    assert np.array_equal(val.view(np.uint16), ref["val"].view(np.uint16))
    # low rank: orthonormal rows and near-optimal truncation error of R
    np.testing.assert_allclose(A @ A.T, np.eye(2), atol=3e-3)
    R = ref["R"]
    opt = np.sum(R ** 2) - np.sum(ref["B"] ** 2)        # error of the exact truncated SVD
    err = np.sum((R - A.T @ B) ** 2)
    assert err <= opt + 2e-3 * np.sum(R ** 2) + 1e-12, (err, opt, np.sum(R ** 2))


@pytest.mark.parametrize("D,bits,chunks", [(128, 4, [300, 1, 1, 40, 3]), (64, 4, [200, 33]),
                                            (128, 2, [150, 20, 20])])
def test_gear_pack_against_oracle(kvc, orc, D, bits, chunks):
    """Bulk and decode-sized appends of a GEAR cache: every flushed group's KIVI blocks and
    sparse parts are bit-exact, its rank-2 factors near-optimal."""
    B_, Hkv, R = 2, 2, 64
    T = sum(chunks)
    g = torch.Generator().manual_seed(D + bits + T)
    K = (torch.randn(B_, Hkv, T, D, generator=g) *
         torch.rand(B_, Hkv, 1, D, generator=g) * 3).half()
    V = torch.randn(B_, Hkv, T, D, generator=g).half()
    n_q = orc.kivi_nq(T, R)
    cache = kvc.QuantCache.empty(B_, Hkv, n_q, D, bits, R, gear=True)
    t0 = 0
    for c in chunks:
        kvc.kvc_append_quant(cache, K[:, :, t0:t0 + c].cuda().contiguous(),
                             V[:, :, t0:t0 + c].cuda().contiguous())
        t0 += c
    torch.cuda.synchronize()
    for b in range(B_):
        for h in range(Hkv):
            gz = gr.quantize_unit(np16(K[b, h, :n_q]), np16(V[b, h, :n_q]), n_q, bits)
            kb, vb = orc.kivi_pack_unit(gz["qz"], D, bits)
            assert np.array_equal(cache.k_blocks[b, h].cpu().numpy(), kb)
            assert np.array_equal(cache.v_blocks[b, h].cpu().numpy(), vb)
            kg, vg = cache.k_gear[b, h].cpu().numpy(), cache.v_gear[b, h].cpu().numpy()
            for gi in range(n_q // G):
                _check_group(kg[gi], gz["k"][gi], D)
                _check_group(vg[gi], gz["v"][gi], D)
    assert device_status_clean(kvc)


def test_gear_pack_ties(kvc, orc):
    """Selections decided by ties, bit-exact against the oracle: groups on the 4-bit grid
    (every residual 0: the sparse part is the first n_s flat indices) and grid groups with 200
    entries moved by exactly +-1/64 (all |e| equal at the threshold: the lowest 82 of them by
    flat index, spread over every warp's range)."""
    D, bits, R = 128, 4, 32
    rng = np.random.default_rng(21)
    td = (np.arange(G)[:, None] + np.arange(D)[None, :]) % 32
    pin = (td == 0) | (td == 1)

    def grid_group(n_moved):
        C = rng.integers(1, 15, (G, D)).astype(np.float64)
        C[td == 0], C[td == 1] = 0, 15
        x = 4.0 * (-1.0 + C / 16.0)
        free = np.flatnonzero(~pin.reshape(-1))
        moved = rng.choice(free, n_moved, replace=False)
        x.reshape(-1)[moved] += rng.choice([-1.0, 1.0], n_moved) / 64
        return x.astype(np.float16)

    groups = [grid_group(0), grid_group(200), grid_group(200), grid_group(0)]
    n_ring = 40
    X = np.concatenate(groups + [(rng.standard_normal((n_ring, D)) - 2).astype(np.float16)])
    K = torch.from_numpy(X)[None, None]
    V = torch.from_numpy(np.ascontiguousarray(X[::-1]))[None, None]   # other tie positions
    T = X.shape[0]
    cache, _ = _build_gear(kvc, K, V, bits, R, 512, [T - 3, 3], [0])
    n_q = kivi_nq(T, R)
    gz = gr.quantize_unit(np16(K[0, 0, :n_q]), np16(V[0, 0, :n_q]), n_q, bits)
    kg, vg = cache.k_gear[0, 0].cpu().numpy(), cache.v_gear[0, 0].cpu().numpy()
    for gi in range(n_q // G):
        for side, ref in ((kg[gi], gz["k"][gi]), (vg[gi], gz["v"][gi])):
            _check_group(side, ref, D)
    assert np.array_equal(gz["k"][0]["idx"].astype(np.int64), np.arange(gr.n_sparse(D)))
    assert device_status_clean(kvc)


def test_gear_ragged_edge_lengths(kvc, orc):
    """GEAR at the edges of the flush rule (empty, one token, R, R + 31, R + 32, R + 33,
    R + 100), one batch, on groups whose values sit on the 4-bit grid: every residual is 0, so
    the corrections vanish and the attention must equal KIVI's (the C oracle's)."""
    from test_gpu_kivi import _check_ragged, _ragged_quant_cache
    D, Hq, Hkv, R, bits = 128, 8, 2, 64, 4
    lens = [0, 1, R, R + 31, R + 32, R + 33, R + 100]
    T = max(lens)
    rng = np.random.default_rng(31)
    td = (np.arange(T)[:, None] + np.arange(D)[None, :]) % 32
    def grid(nb):
        c = rng.integers(0, 16, (nb, Hkv, T, D))
        c[..., td == 0], c[..., td == 1] = 0, 15
        return torch.from_numpy((-1.0 + c / 16.0).astype(np.float16))
    K, V = grid(len(lens)), grid(len(lens))
    q = torch.from_numpy(rng.standard_normal((len(lens), Hq, D))).half()
    cache = _ragged_quant_cache(kvc, K, V, lens, bits, R, 128, gear=True)
    o, lse = _attend(kvc, cache, q.cuda())
    _check_ragged(orc, q, K, V, lens, R, bits, o, lse)
    assert device_status_clean(kvc)


# ------------------------------------------------------------------ decode attention
# Logits carry the KIVI path's binary16 rounding of q * s (see test_gpu_kivi.py) plus the
# rank-2 factors' difference between the GPU's subspace iteration and the oracle's SVD.
GEAR_LSE_TOL = 1e-3


def _build_gear(kvc, Kseq, Vseq, bits, R, Cq, chunks, offsets):
    """GEAR cache of Kseq/Vseq [B, Hkv, T, D] (host): offsets[b] tokens of sequence b placed
    in the residual ring first, then the rest appended in the given chunk sizes."""
    B, Hkv, T, D = Kseq.shape
    cache = kvc.QuantCache.empty(B, Hkv, Cq, D, bits, R, gear=True)
    off = np.asarray(offsets, np.int64)
    for b in range(B):
        for p in range(off[b]):
            cache.k_res[b, :, p % (R + G)] = Kseq[b, :, p].cuda()
            cache.v_res[b, :, p % (R + G)] = Vseq[b, :, p].cuda()
    cache.len.copy_(torch.as_tensor(off, dtype=torch.int32))
    t = 0
    for n_new in chunks:
        kn = torch.stack([Kseq[b, :, off[b] + t:off[b] + t + n_new] for b in range(B)])
        vn = torch.stack([Vseq[b, :, off[b] + t:off[b] + t + n_new] for b in range(B)])
        kvc.kvc_append_quant(cache, kn.cuda().contiguous(), vn.cuda().contiguous())
        t += n_new
    torch.cuda.synchronize()
    return cache, off + t


def _attend(kvc, cache, q, splits=0):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda")
    ws = torch.empty(max(kvc.kvc_workspace_size(cache, q, splits) // 4, 1), dtype=torch.float32,
                     device="cuda")
    kvc.kvc_decode_attend(cache, q, o, lse=lse, workspace=ws, num_splits=splits)
    torch.cuda.synchronize()
    return o, lse


def _oracle_gear_cache(kvc, Kseq, Vseq, lens, bits, R, Cq):
    """A GEAR cache written entirely from the oracle: per unit the KIVI blocks
    (kivi_pack_unit), the side blocks (gear.pack_side of the SVD factors) and the fp16 ring of
    the newest tokens.  Returns the cache and the oracle's per-unit GEAR parts."""
    B, Hkv, T, D = Kseq.shape
    cache = kvc.QuantCache.empty(B, Hkv, Cq, D, bits, R, gear=True)
    parts = {}
    for b in range(B):
        T_b = int(lens[b])
        n_q = kivi_nq(T_b, R)
        for h in range(Hkv):
            Kb, Vb = np16(Kseq[b, h, :T_b]), np16(Vseq[b, h, :T_b])
            gz = gr.quantize_unit(Kb[:n_q], Vb[:n_q], n_q, bits)
            parts[b, h] = gz
            if n_q:
                kb, vb = kivi_pack_unit(gz["qz"], D, bits)
                cache.k_blocks[b, h, :n_q // G] = torch.from_numpy(kb).cuda()
                cache.v_blocks[b, h, :n_q // G] = torch.from_numpy(vb).cuda()
                cache.k_gear[b, h, :n_q // G] = torch.from_numpy(
                    np.stack([gr.pack_side(p, D) for p in gz["k"]])).cuda()
                cache.v_gear[b, h, :n_q // G] = torch.from_numpy(
                    np.stack([gr.pack_side(p, D) for p in gz["v"]])).cuda()
            for t in range(n_q, T_b):
                cache.k_res[b, h, t % (R + G)] = torch.from_numpy(Kb[t]).cuda()
                cache.v_res[b, h, t % (R + G)] = torch.from_numpy(Vb[t]).cuda()
    cache.len.copy_(torch.as_tensor(np.asarray(lens), dtype=torch.int32))
    torch.cuda.synchronize()
    return cache, parts


@pytest.mark.parametrize("D,bits,R,Hq,Hkv,splits", [
    (128, 4, 128, 8, 1, 0), (64, 4, 16, 4, 4, 0), (128, 4, 100, 3, 3, 0), (128, 4, 128, 8, 2, 3),
    (128, 2, 16, 8, 2, 0), (64, 4, 16, 8, 1, 2), (64, 2, 0, 4, 2, 0), (128, 4, 32, 16, 2, 5)])
def test_gear_attention_small(kvc, orc, D, bits, R, Hq, Hkv, splits):
    """Decode attention over GEAR caches written by the oracle (ragged: ring-only, one group
    and many groups; one to several splits; head groups of 1 to 8) against the oracle's
    attention over x_q + S + A^T B of the same parts."""
    g = torch.Generator().manual_seed(11 * D + bits + Hq + R)
    B = 3
    lens = [150, 40 + R, 2 * R + 300]
    T = max(lens)
    Kseq = (torch.randn(B, Hkv, T, D, generator=g) + torch.rand(1, Hkv, 1, D, generator=g) * 4
            - 2).half()
    Vseq = (torch.randn(B, Hkv, T, D, generator=g) + torch.rand(1, Hkv, 1, D, generator=g) * 4
            - 2).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    cache, parts = _oracle_gear_cache(kvc, Kseq, Vseq, lens, bits, R, 1024)
    o, lse = _attend(kvc, cache, q.cuda(), splits)
    gq = Hq // Hkv
    for b in range(B):
        for hk in range(Hkv):
            ref, ref_lse = gr.attend_unit(np16(q[b, hk * gq:(hk + 1) * gq]), np16(Kseq[b, hk]),
                                          np16(Vseq[b, hk]), lens[b], R, bits, gz=parts[b, hk])
            assert_o_close(np16(o[b, hk * gq:(hk + 1) * gq]), ref, what=f"b={b} hk={hk}")
            np.testing.assert_allclose(lse[b, hk * gq:(hk + 1) * gq].cpu().numpy(), ref_lse,
                                       atol=GEAR_LSE_TOL, rtol=0)
    assert device_status_clean(kvc)


def _grid_rank2_tokens(rng, n_groups, D, bits=4, amp=0.2):
    """n_groups 32-token groups whose quantisation residual is dominated by a rank-2 term:
    x = 4 * (-1 + (c + delta) / 2^bits) with codes c; c = 0 and c = cmax = 2^bits - 1 pinned
    where (t + d) % 32 is 0 and 1 (so every K channel and every V token-group of 32 channels
    spans exactly [-4, -4 + 4 cmax / 2^bits]: scale 4 / 2^bits, zero -4), other codes in
    [1, cmax - 1], and delta = amp * (a b^T) for a [32, 2], b [2, D] uniform in [-1, 1]
    (|delta| <= 0.4, zero at the pinned entries).  The residual's third singular value is about
    a third of its second, so its dominant 2-dimensional subspace is well determined."""
    cmax = (1 << bits) - 1
    td = (np.arange(G)[:, None] + np.arange(D)[None, :]) % 32
    pin = (td == 0) | (td == 1)
    out = []
    for _ in range(n_groups):
        C = rng.integers(1, cmax, (G, D)).astype(np.float64)
        C[td == 0], C[td == 1] = 0, cmax
        dl = amp * (rng.uniform(-1, 1, (G, 2)) @ rng.uniform(-1, 1, (2, D)))
        dl[pin] = 0
        out.append(4.0 * (-1.0 + (C + dl) / (cmax + 1)))
    return np.concatenate(out).astype(np.float16)


def _grid_rank2_case(rng, B, Hkv, n_groups, n_ring, D, bits=4):
    """K and V [B, Hkv, 32 n_groups + n_ring, D]: grid + rank-2 groups, then ring tokens."""
    def one():
        return np.concatenate([_grid_rank2_tokens(rng, n_groups, D, bits),
                               (rng.standard_normal((n_ring, D)) - 2).astype(np.float16)])
    K = np.stack([np.stack([one() for _ in range(Hkv)]) for _ in range(B)])
    V = np.stack([np.stack([one() for _ in range(Hkv)]) for _ in range(B)])
    return torch.from_numpy(K), torch.from_numpy(V)


@pytest.mark.parametrize("D,bits,R,chunks", [(128, 4, 64, [300, 1, 19, 57]),
                                             (64, 4, 32, [200, 1, 6]),
                                             (128, 2, 64, [150, 1, 1, 100])])
def test_gear_pack_then_attend(kvc, orc, D, bits, R, chunks):
    """End to end: appends (bulk and decode-sized) pack the GEAR cache on the GPU, then decode
    attention runs over it and must meet the bound against the oracle (its own quantisation,
    sparse selection and SVD).  Groups whose residual has a well-separated rank-2 part (see
    _grid_rank2_tokens) keep the truncated SVD well conditioned, so the GPU's subspace
    iteration must find the same rank-2 term."""
    B, Hkv, Hq = 2, 2, 8
    T = sum(chunks)
    n_q = kivi_nq(T, R)
    rng = np.random.default_rng(D + bits + R)
    Kseq, Vseq = _grid_rank2_case(rng, B, Hkv, n_q // G, T - n_q, D, bits)
    q = torch.from_numpy(rng.standard_normal((B, Hq, D)) * 0.5).half()
    cache, lens = _build_gear(kvc, Kseq, Vseq, bits, R, 512, chunks, [0, 0])
    o, lse = _attend(kvc, cache, q.cuda())
    gq = Hq // Hkv
    for b in range(B):
        for hk in range(Hkv):
            ref, ref_lse = gr.attend_unit(np16(q[b, hk * gq:(hk + 1) * gq]), np16(Kseq[b, hk]),
                                          np16(Vseq[b, hk]), T, R, bits)
            assert_o_close(np16(o[b, hk * gq:(hk + 1) * gq]), ref, what=f"b={b} hk={hk}")
            np.testing.assert_allclose(lse[b, hk * gq:(hk + 1) * gq].cpu().numpy(), ref_lse,
                                       atol=GEAR_LSE_TOL, rtol=0)
    assert device_status_clean(kvc)


def test_gear_corrections_are_applied(kvc, orc):
    """On a unit whose KIVI-4 residual is mostly a rank-2 term, the GPU's GEAR output meets
    the bound against the GEAR oracle, is far from the KIVI oracle, and is much closer than
    KIVI to exact attention over the fp16 values."""
    D, R, Hq = 128, 32, 8
    rng = np.random.default_rng(1)
    n_groups, n_ring = 12, 40
    Kseq, Vseq = _grid_rank2_case(rng, 1, 1, n_groups, n_ring, D)
    T = 32 * n_groups + n_ring
    q = torch.from_numpy(rng.standard_normal((1, Hq, D))).half()
    cache, _ = _build_gear(kvc, Kseq, Vseq, 4, R, 512, [T - 1, 1], [0])
    o, _ = _attend(kvc, cache, q.cuda())
    o = np16(o[0]).astype(np.float64)
    qn, Kn, Vn = np16(q[0]), np16(Kseq[0, 0]), np16(Vseq[0, 0])
    ref_gear, _ = gr.attend_unit(qn, Kn, Vn, T, R, 4)
    ref_kivi, _ = orc.kivi_attend_unit(qn, Kn, Vn, T, R, 4)
    s = (qn.astype(np.float64) @ Kn.astype(np.float64).T) / np.sqrt(D)
    w = np.exp(s - s.max(1, keepdims=True))
    exact = (w / w.sum(1, keepdims=True)) @ Vn.astype(np.float64)
    assert_o_close(o, ref_gear, what="gear")
    e_kivi = np.abs(ref_kivi - exact).mean()
    assert np.abs(o - ref_kivi).max() > 3 * np.abs(o - ref_gear).max()
    assert np.abs(o - exact).mean() < 0.6 * e_kivi, (np.abs(o - exact).mean(), e_kivi)
    assert device_status_clean(kvc)


def test_gear_full_size_sampled(kvc, orc):
    """The heavy GQA workload (B=512, 64 query / 8 KV heads, D=128, T=2048) as a GEAR-4 cache
    packed on the GPU by one bulk append and one decode append.  Sampled units: KIVI blocks and
    sparse parts bit-exact, rank-2 factors near-optimal; their side blocks are then replaced by
    the oracle's (SVD factors) and the attention of the full launch is compared there."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.WORKLOADS["heavy-gqa64x8-b512-d128-t2048"]
    K, V = W.kv_tensors(w, device="cuda")
    q = W.q_tensor(w, device="cuda")
    Cq = orc.kivi_nq(w.T, w.kivi_R)
    cache = kvc.QuantCache.empty(w.B, w.Hkv, Cq, w.D, 4, w.kivi_R, gear=True)
    kvc.kvc_append_quant(cache, K[:, :, :w.T - 1].contiguous(), V[:, :, :w.T - 1].contiguous())
    kvc.kvc_append_quant(cache, K[:, :, w.T - 1:].contiguous(), V[:, :, w.T - 1:].contiguous())
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    gq = w.Hq // w.Hkv
    sample = [(b, int(rng.integers(0, w.Hkv)))
              for b in sorted(set(rng.integers(0, w.B, 3).tolist()) | {w.B - 1})]
    parts = {}
    for b, hk in sample:
        gz = gr.quantize_unit(np16(K[b, hk, :Cq]), np16(V[b, hk, :Cq]), Cq, 4)
        parts[b, hk] = gz
        kb, vb = kivi_pack_unit(gz["qz"], w.D, 4)
        assert np.array_equal(cache.k_blocks[b, hk].cpu().numpy(), kb)
        assert np.array_equal(cache.v_blocks[b, hk].cpu().numpy(), vb)
        kg, vg = cache.k_gear[b, hk].cpu().numpy(), cache.v_gear[b, hk].cpu().numpy()
        for gi in range(0, Cq // G, 7):
            _check_group(kg[gi], gz["k"][gi], w.D)
            _check_group(vg[gi], gz["v"][gi], w.D)
        cache.k_gear[b, hk] = torch.from_numpy(np.stack([gr.pack_side(p, w.D) for p in gz["k"]]))
        cache.v_gear[b, hk] = torch.from_numpy(np.stack([gr.pack_side(p, w.D) for p in gz["v"]]))
    o, lse = _attend(kvc, cache, q)
    for b, hk in sample:
        ref, ref_lse = gr.attend_unit(np16(q[b, hk * gq:(hk + 1) * gq]), np16(K[b, hk]),
                                      np16(V[b, hk]), w.T, w.kivi_R, 4, gz=parts[b, hk])
        assert_o_close(np16(o[b, hk * gq:(hk + 1) * gq]), ref, what=f"b={b} hk={hk}")
        np.testing.assert_allclose(lse[b, hk * gq:(hk + 1) * gq].cpu().numpy(), ref_lse,
                                   atol=GEAR_LSE_TOL, rtol=0)
    assert device_status_clean(kvc)
