"""GPU parity: decode attention over fp16 slot caches vs the fp64 oracle (called via the C ABI)."""
import numpy as np
import pytest
import torch

from helpers import LSE_ABS_TOL, assert_o_close, device_status_clean, np16, slot_cache_from

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def _run(kvc, cache, q, want_logits=False, splits=0):
    B, Hq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    logits = torch.full((B, Hq, cache.C), float("nan"), dtype=torch.float32, device="cuda") \
        if want_logits else None
    ws_bytes = kvc.kvc_workspace_size(cache, q, splits)
    ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device="cuda")
    kvc.kvc_decode_attend(cache, q, o, logits=logits, lse=lse, workspace=ws, num_splits=splits)
    torch.cuda.synchronize()
    return o, lse, logits


@pytest.mark.parametrize("B,Hq,Hkv,C,D,splits", [
    (2, 4, 4, 100, 64, 0), (2, 4, 4, 100, 64, 3), (3, 16, 2, 300, 128, 0),
    (3, 16, 2, 300, 128, 1), (3, 16, 2, 300, 128, 4), (2, 8, 8, 129, 128, 2),
    (1, 8, 1, 513, 128, 0), (2, 6, 2, 70, 64, 2),
    (2, 16, 2, 1024, 128, 8), (1, 8, 1, 1500, 128, 12), (3, 4, 4, 200, 64, 4),
    # more than 32 splits: the combine reads the (m, l) pairs in two rounds of lanes
    (1, 8, 2, 4096, 128, 64), (1, 4, 4, 2560, 64, 40)])
def test_slots_ragged(kvc, orc, B, Hq, Hkv, C, D, splits):
    g = torch.Generator().manual_seed(B * 1000 + C + D + splits)
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    V = torch.randn(B, Hkv, C, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    rng = np.random.default_rng(C + splits)
    n = rng.integers(0, C + 1, size=(B, Hkv))
    n.flat[0] = C
    n.flat[-1] = 1 if n.size > 1 else C
    if n.size > 2:
        n.flat[1] = 0           # an empty unit
    cache = slot_cache_from(kvc, K, V, n, C)
    o, lse, logits = _run(kvc, cache, q.cuda(), want_logits=True, splits=splits)
    ref, ref_lse, ref_lg = orc.decode_attend(np16(q), np16(K), np16(V), n, want_logits=True)
    assert_o_close(np16(o), ref)
    lse_g = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.all(np.isneginf(lse_g[~fin]))
    np.testing.assert_allclose(lse_g[fin], ref_lse[fin], atol=LSE_ABS_TOL, rtol=0)
    lg = logits.cpu().numpy().astype(np.float64)
    gq = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            nn = n[b, h // gq]
            np.testing.assert_allclose(lg[b, h, :nn], ref_lg[b, h, :nn], atol=LSE_ABS_TOL, rtol=0)
            assert np.all(np.isnan(lg[b, h, nn:]))   # nothing written past the valid slots
    assert device_status_clean(kvc)


def test_splits_agree_bitwise_with_each_other_run_to_run(kvc):
    g = torch.Generator().manual_seed(5)
    B, Hq, Hkv, C, D = 4, 16, 2, 700, 128
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    V = torch.randn(B, Hkv, C, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half().cuda()
    cache = slot_cache_from(kvc, K, V, np.full((B, Hkv), C), C)
    a, _, _ = _run(kvc, cache, q, splits=3)
    b, _, _ = _run(kvc, cache, q, splits=3)
    assert torch.equal(a, b)   # deterministic: no atomics in the reduction


def test_binding_descriptor_follows_replaced_fields(kvc, orc):
    """The binding keeps each cache's descriptor between calls; replacing a field (a new
    tensor for n, K and V swapped for other storage) must reach the next call, and in-place
    updates of the same tensors must need no rebuild."""
    g = torch.Generator().manual_seed(11)
    B, Hq, Hkv, C, D = 2, 8, 2, 96, 64
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    V = torch.randn(B, Hkv, C, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    n0 = np.array([[96, 40], [7, 64]])
    cache = slot_cache_from(kvc, K, V, n0, C)

    def check(Kh, Vh, n):
        o, lse, _ = _run(kvc, cache, q.cuda())
        ref_o, ref_lse, _ = orc.decode_attend(np16(q), np16(Kh), np16(Vh), n)
        assert_o_close(np16(o), ref_o)
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, atol=LSE_ABS_TOL, rtol=0)

    check(K, V, n0)
    n1 = np.array([[13, 96], [50, 1]])
    cache.n = torch.as_tensor(n1, dtype=torch.int32).cuda()       # a new tensor
    check(K, V, n1)
    cache.n.copy_(torch.as_tensor(n0, dtype=torch.int32))        # in place, same storage
    check(K, V, n0)
    K2 = torch.randn(B, Hkv, C, D, generator=g).half()
    V2 = torch.randn(B, Hkv, C, D, generator=g).half()
    cache.K, cache.V = K2.cuda(), V2.cuda()                      # other storage
    check(K2, V2, n0)
    assert device_status_clean(kvc)


@pytest.mark.parametrize("wname", ["llama7b-b8-h32-d128-t2048", "heavy-gqa64x8-b512-d128-t2048"])
def test_full_size_sampled_units(kvc, orc, wname):
    """Full-size workloads in the benchmark's launch configuration (automatic splits); the
    oracle checks sampled (sequence, KV head) units."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.WORKLOADS[wname]
    K, V = W.kv_tensors(w, device="cuda")
    q = W.q_tensor(w, device="cuda")
    cache = kvc.SlotCache(K=K, V=V, pos=torch.arange(w.T, dtype=torch.int32, device="cuda")
                          .expand(w.B, w.Hkv, w.T).contiguous(),
                          n=torch.full((w.B, w.Hkv), w.T, dtype=torch.int32, device="cuda"),
                          seqlen=torch.full((w.B,), w.T, dtype=torch.int32, device="cuda"))
    o, lse, _ = _run(kvc, cache, q)
    rng = np.random.default_rng(0)
    bs = sorted(set(rng.integers(0, w.B, 6).tolist()) | {0, w.B - 1})
    g = w.Hq // w.Hkv
    for b in bs:
        hk = int(rng.integers(0, w.Hkv))
        sl = slice(hk * g, (hk + 1) * g)
        ref, ref_lse, _ = orc.decode_attend(np16(q[b:b + 1, sl]), np16(K[b:b + 1, hk:hk + 1]),
                                            np16(V[b:b + 1, hk:hk + 1]),
                                            np.array([[w.T]], np.int32))
        assert_o_close(np16(o[b:b + 1, sl]), ref, what=f"b={b} hk={hk}")
        np.testing.assert_allclose(lse[b, sl].cpu().numpy(), ref_lse[0], atol=LSE_ABS_TOL, rtol=0)
    assert device_status_clean(kvc)


def test_argument_errors_enqueue_nothing(kvc):
    cache = kvc.SlotCache.empty(1, 2, 64, 128)
    q = torch.zeros(1, 2 * 9, 128, dtype=torch.float16, device="cuda")   # 9 heads per KV head
    o = torch.empty_like(q)
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_decode_attend(cache, q, o)
    assert e.value.status == kvc.KVC_ERR_UNSUPPORTED
    q = torch.zeros(1, 3, 128, dtype=torch.float16, device="cuda")       # not a multiple
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_decode_attend(cache, q, torch.empty_like(q))
    assert e.value.status == kvc.KVC_ERR_INVALID_ARG
    q = torch.zeros(1, 2, 128, dtype=torch.float16, device="cuda")
    big = kvc.SlotCache.empty(1, 2, 256, 128)
    with pytest.raises(kvc.KvcError) as e:   # more than one split needs a workspace
        kvc.kvc_decode_attend(big, q, torch.empty_like(q), num_splits=2)
    assert e.value.status == kvc.KVC_ERR_WORKSPACE


@pytest.mark.parametrize("T", [16384, 32768])
def test_long_single_sequence_auto_splits(kvc, orc, T):
    """One sequence of the heavy-load head layout (GQA 64/8, D 128) at long context, in the launch
    configuration of the throughput profile grid (automatic splits): every unit is checked."""
    B, Hq, Hkv, D = 1, 64, 8, 128
    g = torch.Generator().manual_seed(T)
    K = torch.randn(B, Hkv, T, D, generator=g).half()
    V = torch.randn(B, Hkv, T, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    cache = slot_cache_from(kvc, K, V, np.full((B, Hkv), T), T + 8)
    o, lse, _ = _run(kvc, cache, q.cuda())
    ref, ref_lse, _ = orc.decode_attend(np16(q), np16(K), np16(V), np.full((B, Hkv), T, np.int32))
    assert_o_close(np16(o), ref)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, atol=LSE_ABS_TOL, rtol=0)
    assert device_status_clean(kvc)
