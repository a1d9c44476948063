"""GPU parity of the one-launch decode steps (kvc_h2o_decode_step, kvc_stream_decode_step):
append + attention + the method's eviction in one kernel that writes exactly one K/V row.

H2O ("Rethinking KV Cache Compression" guide, §2 and §16 "4 种方法逐步执行": accumulate the
attention and update the keep set): the GPU and the oracle run prompt scoring, eviction to the
budget and then decode steps independently from the same seeded inputs; every step's output,
keep-set and scores agree (a swap between candidates whose oracle scores tie within 1e-6
relative ends the comparison, as the two runs then hold different caches).  At the benchmark's
shape the fused step and the separate launches (kvc_append -> kvc_decode_attend with the fused
score update -> kvc_h2o_evict) hold the same keep-sets, outputs and scores after every step.

StreamingLLM (same sections: sinks plus the recent window): after every step each unit holds
the closed-form window, each slot its token's rows, and the output matches the oracle.
"""
import numpy as np
import pytest
import torch

from helpers import (LSE_ABS_TOL, SCORE_REL_TOL, assert_o_close, device_status_clean, np16,
                     slot_cache_from)
from test_gpu_evict import _check_keep_with_ties, _units

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


@pytest.mark.parametrize("B,Hq,Hkv,D,L,n_heavy,n_recent,steps,decay,C", [
    (1, 4, 4, 64, 64, 8, 8, 32, 0.0, 68),            # the tiny workload's H2O 8+8
    (2, 16, 2, 128, 300, 32, 64, 40, 0.0, 304),       # registers (<= 576 slots)
    (2, 8, 1, 128, 200, 16, 48, 40, 0.99, 204),       # decayed scores
    (1, 16, 4, 128, 1000, 64, 448, 24, 0.0, 1000),    # shared-memory logits (> 576 slots)
    (2, 8, 8, 64, 40, 8, 0, 24, 0.0, 44),             # no recent window: the new token competes
])
def test_h2o_decode_step_free_running(kvc, orc, B, Hq, Hkv, D, L, n_heavy, n_recent, steps,
                                      decay, C):
    g = torch.Generator().manual_seed(L + steps + Hq + 7)
    T1 = L + steps
    budget = n_heavy + n_recent
    Qp = torch.randn(B, Hq, L, D, generator=g).half()
    Kseq = torch.randn(B, Hkv, T1, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, T1, D, generator=g).half()
    qs = torch.randn(steps, B, Hq, D, generator=g).half()
    cache = slot_cache_from(kvc, Kseq[:, :, :L], Vseq[:, :, :L], np.full((B, Hkv), L), C,
                            seqlen=[L] * B)
    scores = torch.zeros(B, Hkv, C, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvc.kvc_h2o_workspace_size(B, Hq, L) // 4, dtype=torch.float32,
                     device="cuda")
    kvc.kvc_h2o_accumulate_prefill(Qp.cuda(), cache.K, scores, ws, L)
    kvc.kvc_h2o_evict(cache, scores, n_heavy, n_recent)
    ref_sc = orc.h2o_prefill_scores(np16(Qp), np16(Kseq[:, :, :L]), L, threads=4)
    st_pos, st_sc = {}, {}
    for b in range(B):
        for hk in range(Hkv):
            pos = np.arange(L, dtype=np.int32)
            keep, _ = orc.h2o_keep(pos, ref_sc[b, hk], L, n_heavy, n_recent)
            st_pos[b, hk], st_sc[b, hk] = pos[keep], ref_sc[b, hk][keep]
    K16, V16 = np16(Kseq), np16(Vseq)
    o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    gq = Hq // Hkv
    compared = 0
    for s_ in range(steps):
        T = L + s_
        kvc.kvc_h2o_decode_step(cache, scores, qs[s_].cuda(), Kseq[:, :, T:T + 1].cuda().contiguous(),
                                Vseq[:, :, T:T + 1].cuda().contiguous(), o, lse, n_heavy, n_recent,
                                decay)
        torch.cuda.synchronize()
        n, pos_g, K_g, V_g = _units(cache)
        assert (cache.seqlen.cpu().numpy() == T + 1).all()
        sc_g = scores.cpu().numpy()
        diverged = False
        for b in range(B):
            for hk in range(Hkv):
                pos = np.concatenate([st_pos[b, hk], [T]]).astype(np.int32)
                sc = np.concatenate([st_sc[b, hk], [0.0]])
                q_u = np16(qs[s_, b, hk * gq:(hk + 1) * gq])[None]
                o_r, lse_r, lg_r = orc.decode_attend(q_u, K16[b, hk][pos][None, None],
                                                     V16[b, hk][pos][None, None],
                                                     np.array([[pos.size]]), want_logits=True)
                assert_o_close(np16(o[b, hk * gq:(hk + 1) * gq]), o_r[0], what=f"step {s_}")
                np.testing.assert_allclose(lse[b, hk * gq:(hk + 1) * gq].cpu().numpy(), lse_r[0],
                                           atol=LSE_ABS_TOL, rtol=0)
                sc = orc.h2o_accumulate(sc[None, None], lg_r, lse_r, np.array([[pos.size]]),
                                        decay=float(np.float32(decay)))[0, 0]
                keep, _ = orc.h2o_keep(pos, sc, T + 1, n_heavy, n_recent)
                nn = n[b, hk]
                got = pos_g[b, hk, :nn]
                assert nn == min(budget, pos.size)
                if _check_keep_with_ties(got, pos, sc, T + 1, n_heavy, n_recent):
                    diverged = True
                else:
                    compared += 1
                    order = np.argsort(got)
                    want = dict(zip(pos.tolist(), sc.tolist()))
                    np.testing.assert_allclose(sc_g[b, hk, :nn][order],
                                               [want[int(p)] for p in got[order]],
                                               rtol=SCORE_REL_TOL)
                    # every kept slot holds its token's K and V rows
                    assert np.array_equal(K_g[b, hk, :nn], K16[b, hk][got].view(np.uint16))
                    assert np.array_equal(V_g[b, hk, :nn], V16[b, hk][got].view(np.uint16))
                st_pos[b, hk], st_sc[b, hk] = pos[keep], sc[keep]
        if diverged:
            break
    assert compared > 0
    assert device_status_clean(kvc)


@pytest.mark.parametrize("B", [64, 512])
def test_h2o_decode_step_matches_separate_launches_bench_shape(kvc, B):
    """The heavy-load shape (GQA 64/8, D 128, 520-slot caches at the 512 budget after a seeded
    prefill state): 24 steps of kvc_h2o_decode_step against the same steps as kvc_append ->
    kvc_decode_attend(h2o_scores) -> kvc_h2o_evict from an identical start, at 64 sequences
    (one launch, 24 steps) and at the benchmark's 512 (more than four units per SM: the call
    issues the three launches itself; 6 steps).  Keep-sets must agree (as sets; near-ties within 1e-6 relative
    may swap), outputs within the fp16 tolerance and scores within 1e-4 relative."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.HEAVY
    Hq, Hkv, D, T0, C = w.Hq, w.Hkv, w.D, w.T, 520
    n_heavy, n_recent, steps = w.n_heavy, w.n_recent, (24 if B <= 64 else 6)
    Kseq, Vseq = W.kv_tensors(w, T=T0 + steps, B=B, device="cuda")
    rng = np.random.default_rng(64)
    pos0 = np.zeros((B, Hkv, 512), np.int32)
    for b in range(B):
        for hk in range(Hkv):
            heavy = np.sort(rng.choice(T0 - n_recent, n_heavy, replace=False))
            pos0[b, hk] = rng.permutation(np.concatenate([heavy, np.arange(T0 - n_recent, T0)]))
    sc0 = torch.from_numpy(rng.uniform(0.0, 4.0, (B, Hkv, 512)).astype(np.float32)).cuda()
    caches, scores = [], []
    for _ in range(2):
        c = kvc.SlotCache.empty(B, Hkv, C, D)
        idx = torch.from_numpy(pos0).long().cuda()[..., None].expand(-1, -1, -1, D)
        c.K[:, :, :512] = torch.gather(Kseq, 2, idx)
        c.V[:, :, :512] = torch.gather(Vseq, 2, idx)
        c.pos[:, :, :512] = torch.from_numpy(pos0).cuda()
        c.n.fill_(512)
        c.seqlen.fill_(T0)
        sc = torch.zeros(B, Hkv, C, dtype=torch.float32, device="cuda")
        sc[:, :, :512] = sc0
        caches.append(c)
        scores.append(sc)
    fused, sep = caches
    o_f = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    o_s = torch.empty_like(o_f)
    lse_f = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    lse_s = torch.empty_like(lse_f)
    for s_ in range(steps):
        q = W.q_tensor(w, B=B, device="cuda", seed_offset=s_)
        kn, vn = Kseq[:, :, T0 + s_:T0 + s_ + 1].contiguous(), Vseq[:, :, T0 + s_:T0 + s_ + 1].contiguous()
        kvc.kvc_h2o_decode_step(fused, scores[0], q, kn, vn, o_f, lse_f, n_heavy, n_recent)
        kvc.kvc_append(sep, kn, vn)
        kvc.kvc_decode_attend(sep, q, o_s, lse=lse_s, num_splits=1, h2o_scores=scores[1])
        kvc.kvc_h2o_evict(sep, scores[1], n_heavy, n_recent)
        torch.cuda.synchronize()
        assert_o_close(np16(o_f).astype(np.float64), np16(o_s).astype(np.float64),
                       what=f"step {s_}")
        assert torch.allclose(lse_f, lse_s, atol=LSE_ABS_TOL, rtol=0)
        nf, pf = fused.n.cpu().numpy(), fused.pos.cpu().numpy()
        ns, ps = sep.n.cpu().numpy(), sep.pos.cpu().numpy()
        assert (nf == 512).all() and (ns == 512).all()
        sf, ss = scores[0].cpu().numpy(), scores[1].cpu().numpy()
        swaps = 0
        for b in range(B):
            for hk in range(Hkv):
                a, z = set(pf[b, hk, :512].tolist()), set(ps[b, hk, :512].tolist())
                if a != z:
                    swaps += 1
                    continue
                ma = dict(zip(pf[b, hk, :512].tolist(), sf[b, hk, :512].tolist()))
                mz = dict(zip(ps[b, hk, :512].tolist(), ss[b, hk, :512].tolist()))
                kk = sorted(ma)
                np.testing.assert_allclose([ma[k] for k in kk], [mz[k] for k in kk],
                                           rtol=SCORE_REL_TOL)
        assert swaps <= max(2, B * Hkv // 256), f"step {s_}: {swaps} units with different keep-sets"
        # the fused cache's rows are its tokens'
        idx = fused.pos[:, :, :512].long()[..., None].expand(B, Hkv, 512, D)
        assert torch.equal(fused.K[:, :, :512], torch.gather(Kseq, 2, idx))
        assert torch.equal(fused.V[:, :, :512], torch.gather(Vseq, 2, idx))
    assert device_status_clean(kvc)


@pytest.mark.parametrize("B,Hq,Hkv,D,T0,n_sink,n_recent,steps,C", [
    (2, 4, 4, 64, 1, 4, 12, 40, 128),       # window grows, then slides
    (2, 8, 2, 128, 20, 0, 8, 30, 64),       # no sinks
    (3, 16, 4, 128, 600, 64, 448, 12, 520),  # the StreamingLLM-512 window
])
def test_stream_decode_step(kvc, orc, B, Hq, Hkv, D, T0, n_sink, n_recent, steps, C):
    g = torch.Generator().manual_seed(T0 + n_recent + 3)
    Kseq = torch.randn(B, Hkv, T0 + steps, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, T0 + steps, D, generator=g).half()
    qs = torch.randn(steps, B, Hq, D, generator=g).half()
    full = slot_cache_from(kvc, Kseq[:, :, :T0], Vseq[:, :, :T0], np.full((B, Hkv), T0),
                           max(C, T0 + 8), seqlen=[T0] * B)
    kvc.kvc_stream_evict(full, n_sink, n_recent)
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    m = min(C, full.C)
    cache.K[:, :, :m] = full.K[:, :, :m]
    cache.V[:, :, :m] = full.V[:, :, :m]
    cache.pos[:, :, :m] = full.pos[:, :, :m]
    cache.n.copy_(full.n)
    cache.seqlen.copy_(full.seqlen)
    o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    for s_ in range(steps):
        P = T0 + s_
        kvc.kvc_stream_decode_step(cache, qs[s_].cuda(), Kseq[:, :, P:P + 1].cuda().contiguous(),
                                   Vseq[:, :, P:P + 1].cuda().contiguous(), o, lse, n_sink,
                                   n_recent)
        torch.cuda.synchronize()
        want = np.flatnonzero(orc.stream_keep(np.arange(P + 1), P + 1, n_sink, n_recent + 1))
        n, pos, K_g, V_g = _units(cache)
        assert (n == len(want)).all(), f"step {s_}"
        assert (cache.seqlen.cpu().numpy() == P + 1).all()
        for b in range(B):
            for h in range(Hkv):
                got = pos[b, h, :len(want)]
                assert np.array_equal(np.sort(got), want), f"step {s_} unit ({b},{h})"
                assert np.array_equal(K_g[b, h, :len(want)], np16(Kseq[b, h])[got].view(np.uint16))
                assert np.array_equal(V_g[b, h, :len(want)], np16(Vseq[b, h])[got].view(np.uint16))
        wi = torch.as_tensor(want).long()
        ref, ref_lse, _ = orc.decode_attend(np16(qs[s_]), np16(Kseq[:, :, wi]), np16(Vseq[:, :, wi]),
                                            np.full((B, Hkv), len(want)))
        assert_o_close(np16(o).astype(np.float64), ref, what=f"step {s_} o")
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, atol=LSE_ABS_TOL, rtol=0)
    assert device_status_clean(kvc)


def test_decode_step_errors(kvc):
    cache = kvc.SlotCache.empty(1, 2, 2048, 128)
    q = torch.zeros(1, 16, 128, dtype=torch.float16, device="cuda")
    kn = torch.zeros(1, 2, 1, 128, dtype=torch.float16, device="cuda")
    sc = torch.zeros(1, 2, 2048, dtype=torch.float32, device="cuda")
    with pytest.raises(kvc.KvcError) as e:          # logits on chip: at most 1024 slots
        kvc.kvc_h2o_decode_step(cache, sc, q, kn, kn, torch.empty_like(q))
    assert e.value.status == kvc.KVC_ERR_UNSUPPORTED
    small = kvc.SlotCache.empty(1, 2, 64, 128)
    with pytest.raises(kvc.KvcError) as e:          # decay outside {0} U (0, 1)
        kvc.kvc_h2o_decode_step(small, sc, q, kn, kn, torch.empty_like(q), decay=1.5)
    assert e.value.status == kvc.KVC_ERR_INVALID_ARG
    # a unit above budget is flagged and keeps its slots
    full = kvc.SlotCache.empty(1, 2, 64, 128)
    full.n.fill_(20)
    full.pos[:, :, :20] = torch.arange(20, dtype=torch.int32, device="cuda")
    full.seqlen.fill_(20)
    kvc.kvc_h2o_decode_step(full, sc[:, :, :64].contiguous(), q, kn, kn, torch.empty_like(q),
                            n_heavy=4, n_recent=8)
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status() & kvc.KVC_DEV_CAPACITY
    assert full.n.cpu().eq(20).all() and full.seqlen.cpu().eq(21).all()
