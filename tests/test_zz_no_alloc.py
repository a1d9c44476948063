"""kvc_decode_attend_noalloc: decode attention for callers that cannot allocate device memory
on their decode path (an engine whose device memory was all handed to its KV-cache pool at
start-up, or a plugin host that forbids cudaMalloc in its enqueue callback because it
synchronises the device).  Its split scratch is a fixed array owned by the library.

Checked here through the C ABI: two calls in a row agree with kvc_decode_attend (which uses a
caller workspace) within the attention tolerance, and shapes that need more scratch than the
fixed array are rejected.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from helpers import assert_o_close, np16, slot_cache_from

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_split_gb300 import build
    build.build()
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def _reference(kvc, cache, q, splits):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda")
    nb = kvc.kvc_workspace_size(cache, q, splits)
    assert 0 < nb <= kvc.KVC_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(nb // 4, dtype=torch.float32, device="cuda")
    kvc.kvc_decode_attend(cache, q, o, lse=lse, workspace=ws, num_splits=splits)
    torch.cuda.synchronize()
    return o, lse


def _twice(kvc, cache, q, splits):
    outs = []
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
        kvc.kvc_decode_attend_noalloc(cache, q, o, lse=lse, num_splits=splits)
        torch.cuda.synchronize()
        outs.append((o, lse))
    return outs


def test_slot_cache_matches_workspace_entry_point(kvc):
    g = torch.Generator().manual_seed(11)
    B, Hq, Hkv, C, D = 4, 16, 2, 700, 128
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    V = torch.randn(B, Hkv, C, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half().cuda()
    n = np.array([[700, 333], [1, 0], [64, 65], [699, 128]])
    cache = slot_cache_from(kvc, K, V, n, C)
    o_ref, lse_ref = _reference(kvc, cache, q, splits=3)
    for o, lse in _twice(kvc, cache, q, splits=3):
        assert_o_close(np16(o), np16(o_ref).astype(np.float64))
        assert torch.equal(torch.isneginf(lse), torch.isneginf(lse_ref))
        fin = torch.isfinite(lse_ref)
        assert torch.allclose(lse[fin], lse_ref[fin], atol=1e-4, rtol=0)


def test_kivi_cache_matches_workspace_entry_point(kvc):
    g = torch.Generator().manual_seed(12)
    B, Hq, Hkv, D, T = 3, 8, 2, 128, 300
    K = torch.randn(B, Hkv, T, D, generator=g).half().cuda()
    V = torch.randn(B, Hkv, T, D, generator=g).half().cuda()
    q = torch.randn(B, Hq, D, generator=g).half().cuda()
    cache = kvc.QuantCache.empty(B, Hkv, 256, D, 4, 32)
    kvc.kvc_append_quant(cache, K, V)
    torch.cuda.synchronize()
    o_ref, lse_ref = _reference(kvc, cache, q, splits=2)
    for o, lse in _twice(kvc, cache, q, splits=2):
        assert_o_close(np16(o), np16(o_ref).astype(np.float64))
        assert torch.allclose(lse, lse_ref, atol=1e-4, rtol=0)


def test_too_much_scratch_is_rejected(kvc):
    B, Hq, Hkv, D = 256, 64, 8, 128
    cache = kvc.QuantCache.empty(B, Hkv, 512, D, 4, 16)
    q = torch.zeros(B, Hq, D, dtype=torch.float16, device="cuda")
    assert kvc.kvc_workspace_size(cache, q, num_splits=4) > kvc.KVC_NOALLOC_SCRATCH_BYTES
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_decode_attend_noalloc(cache, q, torch.empty_like(q), num_splits=4)
    assert e.value.status == kvc.KVC_ERR_WORKSPACE
