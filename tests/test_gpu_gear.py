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
