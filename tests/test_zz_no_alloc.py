"""kvc_decode_attend_noalloc: decode attention for callers that cannot allocate device memory
on their decode path (an engine whose device memory was all handed to its KV-cache pool at
start-up, or a plugin host that forbids cudaMalloc in its enqueue callback because it
synchronises the device).  Its split scratch is a fixed array owned by the library.

Checked here through the C ABI: two calls in a row agree with kvc_decode_attend (which uses a
caller workspace) within the attention tolerance, for split counts that need the scratch
(several splits of plain attention; more than 8 with the fused H2O update, whose 2..8 splits
merge on chip), for automatic and single-split plans, and with the fused H2O score update;
a second call changes neither torch's allocations nor the device's free memory; shapes that
need more scratch than the fixed array are rejected.  This file is collected last on
purpose."""
import gc

import numpy as np
import pytest
import torch

from helpers import SCORE_REL_TOL, assert_o_close, np16, slot_cache_from

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_split_gb300 import build
    build.build()
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def _reference(kvc, cache, q, splits, logits=None, h2o_scores=None, decay=0.0):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda")
    nb = kvc.kvc_workspace_size(cache, q, splits)
    assert nb <= kvc.KVC_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(max(nb // 4, 1), dtype=torch.float32, device="cuda")
    kvc.kvc_decode_attend(cache, q, o, logits=logits, lse=lse, workspace=ws, num_splits=splits,
                          h2o_scores=h2o_scores, h2o_decay=decay)
    torch.cuda.synchronize()
    return o, lse


def _twice(kvc, cache, q, splits, logits=None, scores0=None, decay=0.0):
    outs = []
    for i in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
        sc = None if scores0 is None else scores0.clone()
        torch.cuda.synchronize()
        if i == 1:   # the second call allocates nothing, neither through torch nor the driver
            gc.collect()   # no collection of earlier garbage may free tensors during the call
            gc.disable()
            alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
        try:
            kvc.kvc_decode_attend_noalloc(cache, q, o, logits=logits, lse=lse, num_splits=splits,
                                          h2o_scores=sc, h2o_decay=decay)
            torch.cuda.synchronize()
            if i == 1:
                assert torch.cuda.memory_allocated() == alloc0
                assert torch.cuda.mem_get_info()[0] == free0
        finally:
            gc.enable()
        outs.append((o, lse, sc))
    return outs


def _close(o, lse, o_ref, lse_ref):
    assert_o_close(np16(o), np16(o_ref).astype(np.float64))
    assert torch.equal(torch.isneginf(lse), torch.isneginf(lse_ref))
    fin = torch.isfinite(lse_ref)
    assert torch.allclose(lse[fin], lse_ref[fin], atol=1e-4, rtol=0)


@pytest.mark.parametrize("splits", [12, 0, 1, 3])
def test_slot_cache_matches_workspace_entry_point(kvc, splits):
    g = torch.Generator().manual_seed(11 + splits)
    B, Hq, Hkv, C, D = 4, 16, 2, 1500, 128
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    V = torch.randn(B, Hkv, C, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half().cuda()
    n = np.array([[1500, 333], [1, 0], [64, 65], [1499, 128]])
    cache = slot_cache_from(kvc, K, V, n, C)
    if splits > 1:     # several splits of plain attention: the fixed scratch is used
        assert kvc.kvc_workspace_size(cache, q, splits) > 0
    o_ref, lse_ref = _reference(kvc, cache, q, splits)
    for o, lse, _ in _twice(kvc, cache, q, splits):
        _close(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("splits,with_logits", [(12, True), (2, False), (0, False)])
def test_fused_h2o_scores_match_workspace_entry_point(kvc, splits, with_logits):
    """The fused heavy-hitter score update through the no-alloc entry point: with 12 splits and
    a logits array (scratch used, scores added by a second launch), and with the logits on chip
    and the splits merged in their cluster (no scratch)."""
    g = torch.Generator().manual_seed(21 + splits)
    B, Hq, Hkv, C, D = 3, 32, 4, 1536, 128
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    V = torch.randn(B, Hkv, C, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half().cuda()
    n = np.array([[1536, 700, 1, 0], [1000, 1536, 64, 65], [1535, 2, 900, 1200]])
    cache = slot_cache_from(kvc, K, V, n, C)
    base = torch.rand(B, Hkv, C, generator=g).cuda()
    logits = torch.empty(B, Hq, C, dtype=torch.float32, device="cuda") if with_logits else None
    sc_ref = base.clone()
    o_ref, lse_ref = _reference(kvc, cache, q, splits, logits=logits, h2o_scores=sc_ref,
                                decay=0.99)
    for o, lse, sc in _twice(kvc, cache, q, splits, logits=logits, scores0=base, decay=0.99):
        _close(o, lse, o_ref, lse_ref)
        assert torch.allclose(sc, sc_ref, rtol=SCORE_REL_TOL, atol=0)


def test_kivi_cache_matches_workspace_entry_point(kvc):
    g = torch.Generator().manual_seed(12)
    B, Hq, Hkv, D, T = 3, 8, 2, 128, 300
    K = torch.randn(B, Hkv, T, D, generator=g).half().cuda()
    V = torch.randn(B, Hkv, T, D, generator=g).half().cuda()
    q = torch.randn(B, Hq, D, generator=g).half().cuda()
    cache = kvc.QuantCache.empty(B, Hkv, 256, D, 4, 32)
    kvc.kvc_append_quant(cache, K, V)
    torch.cuda.synchronize()
    assert kvc.kvc_workspace_size(cache, q, 2) > 0
    o_ref, lse_ref = _reference(kvc, cache, q, splits=2)
    for o, lse, _ in _twice(kvc, cache, q, splits=2):
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
