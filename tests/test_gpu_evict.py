"""GPU parity: StreamingLLM, H2O and random eviction (keep-sets bit-exact vs the oracle,
H2O scores within 1e-4 relative, compacted K/V/pos exact) and the append path."""
import numpy as np
import pytest
import torch

from helpers import (SCORE_REL_TOL, assert_o_close, device_status_clean, np16,
                     slot_cache_from)

pytestmark = pytest.mark.gpu
SEED = 0x243F6A8885A308D3


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def _units(cache):
    """Per unit: (pos array of valid slots, K rows, V rows) on the host."""
    n = cache.n.cpu().numpy()
    pos = cache.pos.cpu().numpy()
    K = cache.K.cpu().numpy().view(np.uint16)
    V = cache.V.cpu().numpy().view(np.uint16)
    return n, pos, K, V


def _assert_content(cache, Kseq, Vseq, b, hk, expect_pos):
    """Valid slots of unit (b,hk) hold exactly expect_pos, each with its original K/V row."""
    n, pos, K, V = _units(cache)
    nn = n[b, hk]
    got = pos[b, hk, :nn]
    assert sorted(got.tolist()) == sorted(int(p) for p in expect_pos), f"unit ({b},{hk})"
    ks = Kseq[b, hk].cpu().numpy().view(np.uint16)
    vs = Vseq[b, hk].cpu().numpy().view(np.uint16)
    assert np.array_equal(K[b, hk, :nn], ks[got]) and np.array_equal(V[b, hk, :nn], vs[got])


def test_append_then_capacity(kvc):
    g = torch.Generator().manual_seed(1)
    B, Hkv, C, D = 2, 3, 40, 64
    k1 = torch.randn(B, Hkv, 30, D, generator=g).half().cuda()
    v1 = torch.randn(B, Hkv, 30, D, generator=g).half().cuda()
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    kvc.kvc_append(cache, k1, v1)
    kvc.kvc_append(cache, k1[:, :, :5].contiguous(), v1[:, :, :5].contiguous())
    torch.cuda.synchronize()
    assert cache.n.cpu().eq(35).all() and cache.seqlen.cpu().eq(35).all()
    assert torch.equal(cache.K[:, :, :30], k1) and torch.equal(cache.V[:, :, 30:35], v1[:, :, :5])
    assert cache.pos[0, 0, :35].cpu().tolist() == list(range(35))
    assert device_status_clean(kvc)
    kvc.kvc_append(cache, k1[:, :, :10].contiguous(), v1[:, :, :10].contiguous())   # 45 > 40
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status() & kvc.KVC_DEV_CAPACITY
    assert cache.n.cpu().eq(35).all()     # units left unchanged


@pytest.mark.parametrize("T,n_sink,n_recent", [(2048, 64, 448), (96, 4, 12), (10, 4, 12),
                                               (700, 0, 100)])
def test_stream_prefill_and_decode(kvc, orc, T, n_sink, n_recent):
    g = torch.Generator().manual_seed(T)
    B, Hkv, D = 2, 4, 128
    C = T + 8
    Kseq = torch.randn(B, Hkv, C, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, C, D, generator=g).half()
    cache = slot_cache_from(kvc, Kseq, Vseq, np.full((B, Hkv), T), C, seqlen=[T] * B)
    kvc.kvc_stream_evict(cache, n_sink, n_recent)
    torch.cuda.synchronize()
    keep = orc.stream_keep(np.arange(T), T, n_sink, n_recent)
    for b in range(B):
        for hk in range(Hkv):
            _assert_content(cache, Kseq, Vseq, b, hk, np.flatnonzero(keep))
    # decode: the next token is appended, attended over, then the window slides
    kvc.kvc_append(cache, Kseq[:, :, T:T + 1].cuda().contiguous(), Vseq[:, :, T:T + 1].cuda().contiguous())
    kvc.kvc_stream_evict(cache, n_sink, n_recent)
    torch.cuda.synchronize()
    keep = orc.stream_keep(np.arange(T + 1), T + 1, n_sink, n_recent)
    for b in range(B):
        for hk in range(Hkv):
            _assert_content(cache, Kseq, Vseq, b, hk, np.flatnonzero(keep))
    assert device_status_clean(kvc)


def _check_keep_with_ties(keep_gpu_pos, pos, score_ref, T, n_heavy, n_recent):
    """GPU keep-set == oracle keep-set, except swaps between candidates whose oracle scores
    tie within 1e-6 relative."""
    keep_ref, margin = None, None
    import oracle as orc
    keep_ref, margin = orc.h2o_keep(pos, score_ref, T, n_heavy, n_recent)
    ref_set = set(pos[keep_ref].tolist())
    got_set = set(int(p) for p in keep_gpu_pos)
    if ref_set == got_set:
        return 0
    extra, missing = got_set - ref_set, ref_set - got_set
    sc = {int(p): s for p, s in zip(pos, score_ref)}
    assert len(extra) == len(missing)
    for a, m in zip(sorted(extra, key=lambda p: -sc[p]), sorted(missing, key=lambda p: sc[p])):
        assert abs(sc[a] - sc[m]) <= 1e-6 * max(abs(sc[a]), abs(sc[m])), (a, m, sc[a], sc[m])
    return len(extra)


@pytest.mark.parametrize("B,Hq,Hkv,L,D,n_heavy,n_recent", [
    (1, 4, 4, 64, 64, 8, 8), (2, 8, 2, 300, 128, 16, 40), (1, 16, 2, 1000, 128, 64, 448),
    (2, 4, 4, 130, 64, 200, 8), (1, 8, 1, 1500, 128, 64, 448), (2, 4, 4, 20, 64, 13, 4),
    (1, 8, 2, 512, 128, 32, 64), (3, 6, 3, 384, 64, 20, 30), (1, 2, 1, 129, 128, 16, 16)])
def test_h2o_prefill_scores_and_evict(kvc, orc, B, Hq, Hkv, L, D, n_heavy, n_recent):
    g = torch.Generator().manual_seed(L + Hq)
    C = L + 4
    Qp = torch.randn(B, Hq, L, D, generator=g).half()
    Kseq = torch.randn(B, Hkv, C, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, C, D, generator=g).half()
    cache = slot_cache_from(kvc, Kseq, Vseq, np.full((B, Hkv), L), C, seqlen=[L] * B)
    scores = torch.zeros(B, Hkv, C, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvc.kvc_h2o_workspace_size(B, Hq, L) // 4, dtype=torch.float32, device="cuda")
    kvc.kvc_h2o_accumulate_prefill(Qp.cuda(), cache.K, scores, ws, L)
    torch.cuda.synchronize()
    ref = orc.h2o_prefill_scores(np16(Qp), np16(Kseq), L, threads=4)
    got = scores.cpu().numpy().astype(np.float64)[..., :L]
    np.testing.assert_allclose(got, ref, rtol=SCORE_REL_TOL, atol=0)
    kvc.kvc_h2o_evict(cache, scores, n_heavy, n_recent)
    torch.cuda.synchronize()
    n, pos, _, _ = _units(cache)
    for b in range(B):
        for hk in range(Hkv):
            _check_keep_with_ties(pos[b, hk, :n[b, hk]], np.arange(L, dtype=np.int32), ref[b, hk],
                                  L, n_heavy, n_recent)
            # scores travel with their slots
            sc = scores[b, hk, :n[b, hk]].cpu().numpy()
            np.testing.assert_allclose(sc, ref[b, hk][pos[b, hk, :n[b, hk]]], rtol=SCORE_REL_TOL)
            _assert_content(cache, Kseq, Vseq, b, hk, pos[b, hk, :n[b, hk]])
    assert device_status_clean(kvc)


@pytest.mark.parametrize("B,Hq,Hkv,L,D", [(1, 4, 4, 64, 64), (2, 8, 2, 300, 128),
                                            (1, 8, 1, 1500, 128), (3, 6, 3, 384, 64)])
def test_h2o_prefill_scores_given_row_normalisers(kvc, orc, B, Hq, Hkv, L, D):
    """Prefill scores with the rows' log-sum-exp supplied (as a causal flash-attention forward
    returns it), so only the column-sum pass runs: the oracle's scores and the two-pass
    call's scores, both within the score tolerance."""
    g = torch.Generator().manual_seed(3 * L + D)
    C = L + 4
    Qp = torch.randn(B, Hq, L, D, generator=g).half()
    Kseq = torch.randn(B, Hkv, C, D, generator=g).half()
    # the rows' natural-log normalisers in fp64 from the fp16 inputs, handed over in fp32
    q64 = Qp.double().numpy()
    k64 = np.repeat(Kseq.double().numpy()[:, :, :L], Hq // Hkv, axis=1)
    s = np.einsum("bhid,bhjd->bhij", q64, k64) / np.sqrt(D)
    s = np.where(np.tril(np.ones((L, L), bool)), s, -np.inf)
    m = s.max(-1, keepdims=True)
    lse = (m[..., 0] + np.log(np.exp(s - m).sum(-1))).astype(np.float32)
    ws = torch.empty(kvc.kvc_h2o_workspace_size(B, Hq, L) // 4, dtype=torch.float32, device="cuda")
    kp = Kseq.cuda()
    given = torch.zeros(B, Hkv, C, dtype=torch.float32, device="cuda")
    kvc.kvc_h2o_accumulate_prefill(Qp.cuda(), kp, given, ws, L, lse=torch.from_numpy(lse).cuda())
    both = torch.zeros(B, Hkv, C, dtype=torch.float32, device="cuda")
    kvc.kvc_h2o_accumulate_prefill(Qp.cuda(), kp, both, ws, L)
    torch.cuda.synchronize()
    ref = orc.h2o_prefill_scores(np16(Qp), np16(Kseq), L, threads=4)
    got = given.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(got[..., :L], ref, rtol=SCORE_REL_TOL, atol=0)
    assert (got[..., L:] == 0).all()
    np.testing.assert_allclose(got[..., :L], both.cpu().numpy()[..., :L], rtol=SCORE_REL_TOL,
                               atol=0)
    assert device_status_clean(kvc)


def test_h2o_prefill_full_size_sampled_units(kvc, orc):
    """The prefill score pass at the benchmark's shape and launch (512 sequences, GQA 64/8,
    D=128, a 2047-token causal prompt; the persistent CTAs claim tile pairs dynamically):
    the oracle recomputes sampled (sequence, KV head) units, and conservation (the scores of
    a unit sum to g * L) holds for every unit."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.HEAVY
    B, Hq, Hkv, D, L = w.B, w.Hq, w.Hkv, w.D, w.T - 1
    g = Hq // Hkv
    K, _ = W.kv_tensors(w, T=w.T, B=B, device="cuda")
    kp = K[:, :, :L].contiguous()
    del K
    qp = W.q_tensor(w, B=B, L=L, device="cuda")
    scores = torch.zeros(B, Hkv, L, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvc.kvc_h2o_workspace_size(B, Hq, L) // 4, dtype=torch.float32, device="cuda")
    for _ in range(2):   # the second call reuses the workspace (its counters are re-zeroed)
        scores.zero_()
        kvc.kvc_h2o_accumulate_prefill(qp, kp, scores, ws, L)
    torch.cuda.synchronize()
    assert device_status_clean(kvc)
    total = scores.double().sum(dim=2).cpu().numpy()
    np.testing.assert_allclose(total, g * L, rtol=1e-4)
    rng = np.random.default_rng(7)
    units = sorted({(0, 0), (B - 1, Hkv - 1)} |
                   {(int(b), int(h)) for b, h in zip(rng.integers(0, B, 2), rng.integers(0, Hkv, 2))})
    for b, hk in units:
        ref = orc.h2o_prefill_scores(np16(qp[b:b + 1, hk * g:(hk + 1) * g]),
                                     np16(kp[b:b + 1, hk:hk + 1]), L, threads=8)
        got = scores[b, hk].cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(got, ref[0, 0], rtol=SCORE_REL_TOL, atol=0,
                                   err_msg=f"b={b} hk={hk}")
    # the column-sum pass alone, with the rows' normalisers supplied (here the ones the
    # two-pass call left in its workspace, -lse in log2 units, turned back to natural log)
    lpad = (L + 127) // 128 * 128
    lse = (ws[:B * Hq * lpad].view(B, Hq, lpad)[:, :, :L] * (-np.log(2.0))).contiguous()
    one = torch.zeros_like(scores)
    kvc.kvc_h2o_accumulate_prefill(qp, kp, one, ws, L, lse=lse)
    torch.cuda.synchronize()
    assert device_status_clean(kvc)
    np.testing.assert_allclose(one.double().sum(dim=2).cpu().numpy(), g * L, rtol=1e-4)
    np.testing.assert_allclose(one.cpu().numpy(), scores.cpu().numpy(), rtol=SCORE_REL_TOL,
                               atol=1e-30)


@pytest.mark.parametrize("B,Hq,Hkv,D,mode,splits,decay", [
    (4, 64, 8, 128, "separate", 0, 0.0), (3, 8, 8, 64, "separate", 0, 0.0),
    (4, 64, 8, 128, "fused", 1, 0.0), (3, 8, 8, 64, "fused", 3, 0.0),
    (4, 64, 8, 128, "fused", 1, 0.99), (3, 8, 8, 64, "separate", 0, 0.9),
    (3, 8, 8, 64, "fused", 3, 0.99), (4, 64, 8, 128, "onchip", 0, 0.0),
    (3, 8, 8, 64, "onchip", 1, 0.99), (2, 24, 8, 128, "onchip", 1, 0.0),
    (4, 64, 8, 128, "onchip", 3, 0.0), (3, 8, 8, 64, "onchip", 2, 0.99),
    (2, 64, 8, 128, "fused", 12, 0.0)])
def test_h2o_decode_step(kvc, orc, B, Hq, Hkv, D, mode, splits, decay):
    """One decode step from a seeded post-prefill state: 64 heavy slots from [0, 1600) plus the
    recent 448; append token 2048, attend over 513 slots, accumulate (plain, or the decayed
    activity score with decay lambda), evict back to 512.  Modes: attention then a separate
    accumulate launch; the accumulate fused into the attention (logits written); fused with the
    logits kept on chip (no logits array)."""
    T, n_heavy, n_recent = 2048, 64, 448
    g = torch.Generator().manual_seed(B * Hq)
    rng = np.random.default_rng(B * Hq)
    C = 520
    Kseq = torch.randn(B, Hkv, T + 1, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, T + 1, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    pos0 = np.zeros((B, Hkv, 512), np.int32)
    sc0 = np.zeros((B, Hkv, C), np.float32)
    for b in range(B):
        for hk in range(Hkv):
            heavy = np.sort(rng.choice(T - n_recent, n_heavy, replace=False))
            p = np.concatenate([heavy, np.arange(T - n_recent, T)]).astype(np.int32)
            p = rng.permutation(p)                  # slot order is free
            pos0[b, hk] = p
            sc0[b, hk, :512] = rng.uniform(0.0, 4.0, 512).astype(np.float32)
    pos_t = torch.from_numpy(pos0).long()
    cache.K[:, :, :512] = torch.gather(Kseq, 2, pos_t[..., None].expand(-1, -1, -1, D)).cuda()
    cache.V[:, :, :512] = torch.gather(Vseq, 2, pos_t[..., None].expand(-1, -1, -1, D)).cuda()
    cache.pos[:, :, :512] = torch.from_numpy(pos0).cuda()
    cache.n.fill_(512)
    cache.seqlen.fill_(T)
    scores = torch.from_numpy(sc0).cuda()
    # the step
    kvc.kvc_append(cache, Kseq[:, :, T:].cuda().contiguous(), Vseq[:, :, T:].cuda().contiguous())
    o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    logits = torch.empty(B, Hq, C, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(kvc.kvc_workspace_size(cache, q, splits) // 4, 1), dtype=torch.float32,
                     device="cuda")
    if mode == "fused":   # probabilities added to the scores by the attention launch itself
        kvc.kvc_decode_attend(cache, q.cuda(), o, logits=logits, lse=lse, workspace=ws,
                              num_splits=splits, h2o_scores=scores, h2o_decay=decay)
    elif mode == "onchip":
        kvc.kvc_decode_attend(cache, q.cuda(), o, lse=lse, workspace=ws, num_splits=splits,
                              h2o_scores=scores, h2o_decay=decay)
    else:
        kvc.kvc_decode_attend(cache, q.cuda(), o, logits=logits, lse=lse, workspace=ws,
                              num_splits=splits)
        kvc.kvc_h2o_accumulate_decode(cache, scores, logits, lse, Hq, decay=decay)
    scores_after_acc = scores.clone()
    kvc.kvc_h2o_evict(cache, scores, n_heavy, n_recent)
    torch.cuda.synchronize()
    # oracle from the same seeded state
    pos513 = np.concatenate([pos0, np.full((B, Hkv, 1), T, np.int32)], axis=2)
    Kc = np.take_along_axis(np16(Kseq), pos513[..., None].astype(np.int64), axis=2)
    Vc = np.take_along_axis(np16(Vseq), pos513[..., None].astype(np.int64), axis=2)
    ref_o, ref_lse, ref_lg = orc.decode_attend(np16(q), Kc, Vc, np.full((B, Hkv), 513),
                                               want_logits=True)
    assert_o_close(np16(o), ref_o)
    sc_ref = np.concatenate([sc0[..., :512].astype(np.float64), np.zeros((B, Hkv, 1))], axis=2)
    sc_ref = orc.h2o_accumulate(sc_ref, ref_lg, ref_lse, np.full((B, Hkv), 513),
                                decay=float(np.float32(decay)))
    np.testing.assert_allclose(scores_after_acc.cpu().numpy()[..., :513], sc_ref,
                               rtol=SCORE_REL_TOL)
    n, pos, _, _ = _units(cache)
    assert (n == 512).all()
    assert (scores[:, :, 512:].cpu() == 0).all()     # the freed slot starts from zero
    for b in range(B):
        for hk in range(Hkv):
            _check_keep_with_ties(pos[b, hk, :512], pos513[b, hk], sc_ref[b, hk], T + 1, n_heavy,
                                  n_recent)
            _assert_content(cache, Kseq, Vseq, b, hk, pos[b, hk, :512])
    assert device_status_clean(kvc)


@pytest.mark.parametrize("C", [517, 520])           # scalar rows / 16-byte rows
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (64, 8), (32, 2)])
@pytest.mark.parametrize("decay", [0.0, 0.9])
def test_h2o_accumulate_decode_layouts(kvc, orc, C, Hq, Hkv, decay):
    """The standalone decode score update against the oracle's definition (H2O: the step's
    attention probabilities summed over the group's query heads), for both row layouts,
    groups of 1, 8 and 16 heads, ragged slot counts (0, C, and values off a multiple of 4),
    plain and decayed scores; slots at or past n keep their old score bit for bit."""
    rng = np.random.default_rng(SEED + C + 7 * Hq)
    B = 3
    logits = rng.normal(0.0, 3.0, (B, Hq, C)).astype(np.float32)
    lse = (np.log(np.exp(logits.astype(np.float64)).sum(-1)) + rng.uniform(0, 2, (B, Hq)))
    lse = lse.astype(np.float32)
    sc0 = rng.uniform(0.0, 4.0, (B, Hkv, C)).astype(np.float32)
    n = rng.integers(0, C + 1, (B, Hkv)).astype(np.int32)
    n.flat[0], n.flat[-1] = 0, C
    n.flat[1 % n.size] = C - 1
    cache = kvc.SlotCache.empty(B, Hkv, C, 64)
    cache.n.copy_(torch.from_numpy(n))
    scores = torch.from_numpy(sc0).cuda()
    kvc.kvc_h2o_accumulate_decode(cache, scores, torch.from_numpy(logits).cuda(),
                                  torch.from_numpy(lse).cuda(), Hq, decay=decay)
    got = scores.cpu().numpy()
    ref = orc.h2o_accumulate(sc0.astype(np.float64), logits, lse, n,
                             decay=float(np.float32(decay)))
    for b in range(B):
        for hk in range(Hkv):
            k = n[b, hk]
            np.testing.assert_allclose(got[b, hk, :k], ref[b, hk, :k], rtol=SCORE_REL_TOL)
            assert np.array_equal(got[b, hk, k:].view(np.uint32), sc0[b, hk, k:].view(np.uint32))
    assert device_status_clean(kvc)


@pytest.mark.parametrize("B,Hq,Hkv,D,L,n_heavy,n_recent,steps,onchip,decay", [
    (1, 4, 4, 64, 64, 8, 8, 32, True, 0.0),          # the tiny workload's H2O 8+8
    (2, 16, 2, 128, 300, 32, 64, 40, False, 0.0),
    (2, 8, 1, 128, 200, 16, 48, 40, True, 0.99)])
def test_h2o_free_running_decode(kvc, orc, B, Hq, Hkv, D, L, n_heavy, n_recent, steps, onchip,
                                 decay):
    """GPU and oracle run the whole H2O life independently from the same seeded inputs: prompt
    score pass, eviction to the budget, then `steps` decode steps of append -> attention with
    the fused score update -> eviction.  Every step's outputs, keep-sets and scores agree; a
    swap between near-tied candidates (accepted) ends the comparison, since the two runs then
    hold different caches."""
    g = torch.Generator().manual_seed(L + steps + Hq)
    T1 = L + steps
    C = L + 4
    budget = n_heavy + n_recent
    Qp = torch.randn(B, Hq, L, D, generator=g).half()
    Kseq = torch.randn(B, Hkv, T1, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, T1, D, generator=g).half()
    qs = torch.randn(steps, B, Hq, D, generator=g).half()
    # ---- GPU
    cache = slot_cache_from(kvc, Kseq[:, :, :L], Vseq[:, :, :L], np.full((B, Hkv), L), C,
                            seqlen=[L] * B)
    scores = torch.zeros(B, Hkv, C, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvc.kvc_h2o_workspace_size(B, Hq, L) // 4, dtype=torch.float32, device="cuda")
    kvc.kvc_h2o_accumulate_prefill(Qp.cuda(), cache.K, scores, ws, L)
    kvc.kvc_h2o_evict(cache, scores, n_heavy, n_recent)
    # ---- oracle state per unit: positions and scores of the kept slots
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
    logits = None if onchip else torch.empty(B, Hq, C, dtype=torch.float32, device="cuda")
    gq = Hq // Hkv
    for s_ in range(steps):
        T = L + s_
        kvc.kvc_append(cache, Kseq[:, :, T:T + 1].cuda().contiguous(),
                       Vseq[:, :, T:T + 1].cuda().contiguous())
        kvc.kvc_decode_attend(cache, qs[s_].cuda(), o, logits=logits, lse=lse, num_splits=1,
                              h2o_scores=scores, h2o_decay=decay)
        kvc.kvc_h2o_evict(cache, scores, n_heavy, n_recent)
        torch.cuda.synchronize()
        n, pos_g, _, _ = _units(cache)
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
                sc = orc.h2o_accumulate(sc[None, None], lg_r, lse_r, np.array([[pos.size]]),
                                        decay=float(np.float32(decay)))[0, 0]
                keep, _ = orc.h2o_keep(pos, sc, T + 1, n_heavy, n_recent)
                got = pos_g[b, hk, :n[b, hk]]
                assert n[b, hk] == budget
                if _check_keep_with_ties(got, pos, sc, T + 1, n_heavy, n_recent):
                    diverged = True
                else:
                    order = np.argsort(got)
                    want = dict(zip(pos.tolist(), sc.tolist()))
                    np.testing.assert_allclose(sc_g[b, hk, :n[b, hk]][order],
                                               [want[int(p)] for p in got[order]],
                                               rtol=SCORE_REL_TOL)
                st_pos[b, hk], st_sc[b, hk] = pos[keep], sc[keep]
        if diverged:
            break
    assert device_status_clean(kvc)


def test_stream_decode_step_full_size_sampled_units(kvc, orc):
    """One StreamingLLM-512 decode step at the benchmark's shape (512 sequences, 8 KV heads,
    a 520-slot cache holding 64 sinks + 448 recent tokens of a 2048-token history in scrambled
    slot order): append, then eviction back to 512 with the one-warp-per-unit kernel.  Every
    unit's keep-set against the closed form, sampled units' rows against their tokens."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.HEAVY
    B, Hkv, D, T, C, n_sink, n_recent = w.B, w.Hkv, w.D, w.T, 520, 64, 448
    rng = np.random.default_rng(512)
    Kseq, Vseq = W.kv_tensors(w, T=T + 1, B=B, device="cuda")
    base = np.concatenate([np.arange(n_sink), np.arange(T - n_recent, T)]).astype(np.int32)
    pos0 = np.stack([np.stack([rng.permutation(base) for _ in range(Hkv)]) for _ in range(B)])
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    idx = torch.from_numpy(pos0).long().cuda()[..., None].expand(-1, -1, -1, D)
    cache.K[:, :, :512] = torch.gather(Kseq, 2, idx)
    cache.V[:, :, :512] = torch.gather(Vseq, 2, idx)
    cache.pos[:, :, :512] = torch.from_numpy(pos0).cuda()
    cache.n.fill_(512)
    cache.seqlen.fill_(T)
    kvc.kvc_append(cache, Kseq[:, :, T:T + 1].contiguous(), Vseq[:, :, T:T + 1].contiguous())
    kvc.kvc_stream_evict(cache, n_sink, n_recent)
    torch.cuda.synchronize()
    assert device_status_clean(kvc)
    assert (cache.n.cpu().numpy() == 512).all()
    want = np.flatnonzero(orc.stream_keep(np.arange(T + 1), T + 1, n_sink, n_recent))
    got = np.sort(cache.pos[:, :, :512].cpu().numpy(), axis=2)
    assert (got == want[None, None, :]).all()
    for b, hk in [(0, 0), (B - 1, Hkv - 1), (int(rng.integers(B)), int(rng.integers(Hkv)))]:
        p = torch.from_numpy(cache.pos[b, hk, :512].cpu().numpy()).long().cuda()
        assert torch.equal(cache.K[b, hk, :512], Kseq[b, hk, p])
        assert torch.equal(cache.V[b, hk, :512], Vseq[b, hk, p])


def test_h2o_decode_step_full_size_sampled_units(kvc, orc):
    """One H2O-512 decode step at the benchmark's shape and launch (512 sequences, GQA 64/8,
    D=128, a 520-slot cache holding 64 heavy + 448 recent tokens of a 2048-token history):
    append, attention with the score update fused and the logits in registers, eviction back
    to 512.  Sampled units against the oracle: outputs, lse, scores and keep-sets."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.HEAVY
    B, Hq, Hkv, D, T, C = w.B, w.Hq, w.Hkv, w.D, w.T, 520
    n_heavy, n_recent = 64, 448
    rng = np.random.default_rng(2048)
    Kseq, Vseq = W.kv_tensors(w, T=T + 1, B=B, device="cuda")
    q = W.q_tensor(w, B=B, device="cuda")
    pos0 = np.empty((B, Hkv, 512), np.int32)
    for b in range(B):
        for hk in range(Hkv):
            heavy = rng.choice(T - n_recent, n_heavy, replace=False)
            pos0[b, hk] = rng.permutation(np.concatenate([heavy, np.arange(T - n_recent, T)]))
    sc0 = rng.uniform(0.0, 4.0, (B, Hkv, C)).astype(np.float32)
    sc0[..., 512:] = 0.0
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    idx = torch.from_numpy(pos0).long().cuda()[..., None].expand(-1, -1, -1, D)
    cache.K[:, :, :512] = torch.gather(Kseq, 2, idx)
    cache.V[:, :, :512] = torch.gather(Vseq, 2, idx)
    cache.pos[:, :, :512] = torch.from_numpy(pos0).cuda()
    cache.n.fill_(512)
    cache.seqlen.fill_(T)
    scores = torch.from_numpy(sc0).cuda()
    kvc.kvc_append(cache, Kseq[:, :, T:T + 1].contiguous(), Vseq[:, :, T:T + 1].contiguous())
    o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    kvc.kvc_decode_attend(cache, q, o, lse=lse, num_splits=1, h2o_scores=scores)
    sc_mid = scores.clone()
    kvc.kvc_h2o_evict(cache, scores, n_heavy, n_recent)
    torch.cuda.synchronize()
    assert device_status_clean(kvc)
    n = cache.n.cpu().numpy()
    assert (n == 512).all()
    g = Hq // Hkv
    pos513 = np.concatenate([pos0, np.full((B, Hkv, 1), T, np.int32)], axis=2)
    for b, hk in sorted({(0, 0), (B - 1, Hkv - 1)} |
                        {(int(x), int(y)) for x, y in zip(rng.integers(0, B, 4),
                                                          rng.integers(0, Hkv, 4))}):
        p = pos513[b, hk]
        Ku = np16(Kseq[b:b + 1, hk:hk + 1, p])
        Vu = np16(Vseq[b:b + 1, hk:hk + 1, p])
        sl = slice(hk * g, (hk + 1) * g)
        ref_o, ref_lse, ref_lg = orc.decode_attend(np16(q[b:b + 1, sl]), Ku, Vu,
                                                   np.array([[513]], np.int32), want_logits=True)
        assert_o_close(np16(o[b:b + 1, sl]), ref_o, what=f"b={b} hk={hk}")
        np.testing.assert_allclose(lse[b, sl].cpu().numpy(), ref_lse[0], atol=1e-4, rtol=0)
        ref_sc = orc.h2o_accumulate(sc0[b:b + 1, hk:hk + 1, :513].astype(np.float64), ref_lg,
                                    ref_lse, np.array([[513]], np.int32))[0, 0]
        np.testing.assert_allclose(sc_mid[b, hk, :513].cpu().numpy(), ref_sc,
                                   rtol=SCORE_REL_TOL, err_msg=f"b={b} hk={hk}")
        got_pos = cache.pos[b, hk, :512].cpu().numpy()
        _check_keep_with_ties(got_pos, p, ref_sc, T + 1, n_heavy, n_recent)
        rows = {int(x): i for i, x in enumerate(p)}
        src = torch.tensor([rows[int(x)] for x in got_pos], device="cuda")
        assert torch.equal(cache.K[b, hk, :512], Kseq[b, hk, torch.from_numpy(p).long().cuda()][src])


@pytest.mark.parametrize("D,C,Hq,Hkv,decay,splits", [
    (128, 576, 64, 8, 0.0, 1), (64, 300, 24, 8, 0.99, 1), (128, 65, 8, 2, 0.0, 1),
    (128, 1500, 64, 8, 0.0, 3),     # three splits of <= 9 tiles: registers, cluster merge
    (64, 2048, 16, 4, 0.99, 2),     # two splits of 16 tiles: shared memory, cluster merge
    (128, 4000, 8, 2, 0.0, 0)])     # automatic plan (at least 4 splits for the on-chip bound)
def test_h2o_register_logits_ragged_vs_oracle(kvc, orc, D, C, Hq, Hkv, decay, splits):
    """The fused H2O launch with the logits kept on chip (registers for splits of up to nine
    tiles, else shared memory; the splits of a unit merged in their cluster) on ragged units
    (empty, one slot, a partial tile, full capacity) and g < 8 query heads per KV head:
    outputs, lse and scores against the oracle's attention and accumulation."""
    B = 3
    g = torch.Generator().manual_seed(C + Hq + D)
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    V = torch.randn(B, Hkv, C, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    rng = np.random.default_rng(C)
    n = rng.integers(0, C + 1, (B, Hkv))
    n[0, 0], n[-1, -1] = 0, C
    n[1, 0] = 1
    cache = slot_cache_from(kvc, K, V, n, C)
    base = torch.rand(B, Hkv, C, generator=g)
    sc = base.clone().cuda()
    o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    kvc.kvc_decode_attend(cache, q.cuda(), o, lse=lse, num_splits=splits, h2o_scores=sc,
                          h2o_decay=decay)
    torch.cuda.synchronize()
    ref_o, ref_lse, ref_lg = orc.decode_attend(np16(q), np16(K), np16(V), n, want_logits=True)
    assert_o_close(np16(o), ref_o)
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse.cpu().numpy()[fin], ref_lse[fin], atol=1e-4, rtol=0)
    ref_sc = orc.h2o_accumulate(base.numpy(), ref_lg, ref_lse, n, decay)
    got = sc.cpu().numpy().astype(np.float64)
    for b in range(B):
        for hk in range(Hkv):
            nn = int(n[b, hk])
            np.testing.assert_allclose(got[b, hk, :nn], ref_sc[b, hk, :nn], rtol=SCORE_REL_TOL,
                                       err_msg=f"b={b} hk={hk}")
            assert np.array_equal(got[b, hk, nn:], base.numpy()[b, hk, nn:])   # untouched
    assert device_status_clean(kvc)


@pytest.mark.parametrize("D,C,n,splits", [(128, 520, 513, 1), (64, 1024, 1024, 1),
                                          (128, 1024, 700, 1), (128, 1500, 1400, 3),
                                          (64, 2048, 2000, 2)])
def test_h2o_onchip_logits_match_written_logits(kvc, D, C, n, splits):
    """The fused H2O launch with the logits kept on chip gives bit-identical outputs, lse and
    scores to the same launch writing a logits array (same arithmetic, other storage), up to
    the on-chip capacity bound."""
    B, Hq, Hkv = 3, 64, 8
    g = torch.Generator().manual_seed(C + n)
    K = torch.randn(B, Hkv, n, D, generator=g).half()
    V = torch.randn(B, Hkv, n, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half().cuda()
    cache = slot_cache_from(kvc, K, V, np.full((B, Hkv), n), C)
    base = torch.rand(B, Hkv, C, generator=g).cuda()
    outs = []
    for onchip in (False, True):
        o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
        lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
        sc = base.clone()
        logits = None if onchip else torch.empty(B, Hq, C, dtype=torch.float32, device="cuda")
        kvc.kvc_decode_attend(cache, q, o, logits=logits, lse=lse, num_splits=splits,
                              h2o_scores=sc, h2o_decay=0.99)
        torch.cuda.synchronize()
        outs.append((o, lse, sc))
    for a, b_ in zip(*outs):
        assert torch.equal(a, b_)
    assert device_status_clean(kvc)


@pytest.mark.parametrize("n_heavy", [9, 0])
def test_h2o_single_drop_cases(kvc, orc, n_heavy):
    """Units that drop exactly one slot (the decode step's case, a path of its own in the
    warp-per-unit kernel): the victim in a middle slot, in the last slot (nothing moves), in
    slot 0, and two candidates tied on the lowest score (the later position leaves); with
    n_heavy = 0 the single candidate leaves.  Keep-sets equal the oracle's exactly, rows and
    scores travel with their positions, and the freed slot's score is 0."""
    B, Hkv, C, D, T, n_recent = 1, 4, 64, 64, 100, 30
    rng = np.random.default_rng(41 + n_heavy)
    g = torch.Generator().manual_seed(41)
    Kseq = torch.randn(B, Hkv, T, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, T, D, generator=g).half()
    n = n_heavy + 1 + n_recent
    pos0 = np.zeros((B, Hkv, C), np.int32)
    sc0 = np.zeros((B, Hkv, C), np.float32)
    for hk in range(Hkv):
        cand = np.sort(rng.choice(T - n_recent, n_heavy + 1, replace=False))
        p = rng.permutation(np.concatenate([cand, np.arange(T - n_recent, T)])).astype(np.int32)
        s = rng.uniform(1.0, 4.0, n).astype(np.float32)
        cslots = np.flatnonzero(p < T - n_recent)
        victim = {0: cslots[len(cslots) // 2], 1: n - 1, 2: cslots[-1], 3: 0}[hk]
        if p[victim] >= T - n_recent:   # bring a candidate into the chosen slot
            o = cslots[0]
            p[[victim, o]] = p[[o, victim]]
            s[[victim, o]] = s[[o, victim]]
        s[victim] = 0.5
        if hk == 2 and n_heavy > 0:     # a tie on the lowest score with another candidate
            other = [c for c in np.flatnonzero(p < T - n_recent) if c != victim][0]
            s[other] = 0.5
        pos0[0, hk, :n], sc0[0, hk, :n] = p, s
    pos_t = torch.from_numpy(pos0).long()
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    cache.K.copy_(torch.gather(Kseq, 2, pos_t[..., None].expand(-1, -1, -1, D)).cuda())
    cache.V.copy_(torch.gather(Vseq, 2, pos_t[..., None].expand(-1, -1, -1, D)).cuda())
    cache.pos.copy_(torch.from_numpy(pos0).cuda())
    cache.n.fill_(n)
    cache.seqlen.fill_(T)
    scores = torch.from_numpy(sc0).cuda()
    kvc.kvc_h2o_evict(cache, scores, n_heavy, n_recent)
    torch.cuda.synchronize()
    nn, pos, _, _ = _units(cache)
    sc = scores.cpu().numpy()
    for hk in range(Hkv):
        assert nn[0, hk] == n - 1
        keep, _ = orc.h2o_keep(pos0[0, hk, :n], sc0[0, hk, :n].astype(np.float64), T, n_heavy,
                               n_recent)
        assert set(pos[0, hk, :n - 1].tolist()) == set(pos0[0, hk, :n][keep].tolist()), hk
        _assert_content(cache, Kseq, Vseq, 0, hk, pos[0, hk, :n - 1])
        src = {int(q): v for q, v in zip(pos0[0, hk, :n], sc0[0, hk, :n])}
        assert all(sc[0, hk, j] == src[int(pos[0, hk, j])] for j in range(n - 1))
        assert sc[0, hk, n - 1] == 0
    assert device_status_clean(kvc)


@pytest.mark.parametrize("C", [600, 1100])   # warp-per-unit and CTA-per-unit kernels
def test_h2o_evict_when_trigger(kvc, orc, C):
    """Batched H2O eviction ("Practical Online KV Cache Compaction for LLM Agents", §5.2): units
    at or above the trigger (here 563 = 110% of a 512 budget) compact to 64 heavy + 448 recent
    exactly as kvc_h2o_evict would; units below it stay bit-identical."""
    B, Hkv, D, T = 2, 4, 128, 3000
    n_heavy, n_recent, trigger = 64, 448, 563
    counts = np.array([[512, 562, 563, 600], [570, 540, 563, 513]], np.int32)
    rng = np.random.default_rng(563)
    g = torch.Generator().manual_seed(563)
    Kseq = torch.randn(B, Hkv, T, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, T, D, generator=g).half()
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    pos0 = np.zeros((B, Hkv, C), np.int32)
    sc0 = np.zeros((B, Hkv, C), np.float32)
    for b in range(B):
        for hk in range(Hkv):
            nn = counts[b, hk]
            heavy = np.sort(rng.choice(T - n_recent, nn - n_recent, replace=False))
            p = rng.permutation(np.concatenate([heavy, np.arange(T - n_recent, T)]))
            pos0[b, hk, :nn] = p
            sc0[b, hk, :nn] = rng.uniform(0.0, 4.0, nn).astype(np.float32)
    pos_t = torch.from_numpy(pos0).long()
    cache.K.copy_(torch.gather(Kseq, 2, pos_t[..., None].expand(-1, -1, -1, D)).cuda())
    cache.V.copy_(torch.gather(Vseq, 2, pos_t[..., None].expand(-1, -1, -1, D)).cuda())
    cache.pos.copy_(torch.from_numpy(pos0).cuda())
    cache.n.copy_(torch.from_numpy(counts).cuda())
    cache.seqlen.fill_(T)
    scores = torch.from_numpy(sc0).cuda()
    K_before, V_before = cache.K.clone(), cache.V.clone()
    kvc.kvc_h2o_evict_when(cache, scores, n_heavy, n_recent, trigger)
    torch.cuda.synchronize()
    n, pos, _, _ = _units(cache)
    sc = scores.cpu().numpy()
    for b in range(B):
        for hk in range(Hkv):
            nn = counts[b, hk]
            if nn < trigger:
                assert n[b, hk] == nn
                assert np.array_equal(pos[b, hk], pos0[b, hk])
                assert np.array_equal(sc[b, hk], sc0[b, hk])
                assert torch.equal(cache.K[b, hk], K_before[b, hk])
                assert torch.equal(cache.V[b, hk], V_before[b, hk])
            else:
                assert n[b, hk] == n_heavy + n_recent
                _check_keep_with_ties(pos[b, hk, :512], pos0[b, hk, :nn],
                                      sc0[b, hk, :nn].astype(np.float64), T, n_heavy, n_recent)
                _assert_content(cache, Kseq, Vseq, b, hk, pos[b, hk, :512])
                assert (sc[b, hk, 512:] == 0).all()
                order = np.argsort(pos[b, hk, :512])
                src = {int(p): s for p, s in zip(pos0[b, hk, :nn], sc0[b, hk, :nn])}
                assert np.array_equal(sc[b, hk, :512][order],
                                      np.array([src[int(p)] for p in pos[b, hk, :512][order]],
                                               np.float32))
    assert device_status_clean(kvc)


def test_random_tiny_two_evictions(kvc, orc):
    """Tiny workload: prompt 64 tokens with the first 16 locked, keep 0.5; evict after the prompt
    (48 candidates -> 24), then after 32 more tokens (56 -> 28)."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.TINY
    B, Hkv, D, C = w.B, w.Hkv, w.D, 128
    Kseq, Vseq = W.kv_tensors(w, T=96)
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    kvc.kvc_append(cache, Kseq[:, :, :64].cuda().contiguous(), Vseq[:, :, :64].cuda().contiguous())
    kvc.kvc_random_evict(cache, w.prompt_len, w.keep_ratio, SEED, 0)
    torch.cuda.synchronize()
    _, pos, _, _ = _units(cache)
    expect = {}
    for hk in range(Hkv):
        keep = orc.random_keep(np.arange(64), w.prompt_len, w.keep_ratio, SEED, 0, 0, hk)
        expect[hk] = np.flatnonzero(keep)
        assert len(expect[hk]) == 16 + 24
        _assert_content(cache, Kseq, Vseq, 0, hk, expect[hk])
    sets = [frozenset(expect[h].tolist()) for h in range(Hkv)]
    assert len(set(sets)) == Hkv              # per-head draws differ; no union
    kvc.kvc_append(cache, Kseq[:, :, 64:96].cuda().contiguous(), Vseq[:, :, 64:96].cuda().contiguous())
    kvc.kvc_random_evict(cache, w.prompt_len, w.keep_ratio, SEED, 1)
    torch.cuda.synchronize()
    n, pos, _, _ = _units(cache)
    for hk in range(Hkv):
        p1 = np.concatenate([expect[hk], np.arange(64, 96)]).astype(np.int32)
        keep = orc.random_keep(p1, w.prompt_len, w.keep_ratio, SEED, 1, 0, hk)
        assert n[0, hk] == 16 + 28
        _assert_content(cache, Kseq, Vseq, 0, hk, p1[keep])
    assert device_status_clean(kvc)


def test_random_reasoning_cadence(kvc, orc):
    """Reasoning-trace workload shape (GQA 64/8, D 128, locked prompt 1024): three evictions
    every 1024 generated tokens at keep 0.25 -> per head 1024 + 256, + 320, + 336 slots."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.REASONING
    B, Hkv, D = 4, w.Hkv, w.D
    steps = 3
    T_all = 1024 + 1024 * steps
    Kseq, Vseq = W.kv_tensors(w, T=T_all, B=B)
    C = 2048 + 512
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    kvc.kvc_append(cache, Kseq[:, :, :2048].cuda().contiguous(), Vseq[:, :, :2048].cuda().contiguous())
    cur = {(b, h): np.arange(2048, dtype=np.int32) for b in range(B) for h in range(Hkv)}
    for e in range(steps):
        if e > 0:
            t0 = 1024 + 1024 * e
            kvc.kvc_append(cache, Kseq[:, :, t0:t0 + 1024].cuda().contiguous(),
                           Vseq[:, :, t0:t0 + 1024].cuda().contiguous())
            for k in cur:
                cur[k] = np.concatenate([cur[k], np.arange(t0, t0 + 1024, dtype=np.int32)])
        kvc.kvc_random_evict(cache, 1024, 0.25, SEED, e)
        torch.cuda.synchronize()
        for (b, h), p in cur.items():
            keep = orc.random_keep(p, 1024, 0.25, SEED, e, b, h)
            cur[(b, h)] = p[keep]
        n, _, _, _ = _units(cache)
        assert (n == 1024 + [256, 320, 336][e]).all()
    for b in range(B):
        for h in range(Hkv):
            _assert_content(cache, Kseq, Vseq, b, h, cur[(b, h)])
    assert device_status_clean(kvc)


def test_random_ratio_one_and_empty_candidates(kvc):
    g = torch.Generator().manual_seed(3)
    B, Hkv, C, D = 1, 2, 64, 64
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    cache = slot_cache_from(kvc, K, K, np.full((B, Hkv), 40), C, seqlen=[40])
    before = cache.K.clone()
    kvc.kvc_random_evict(cache, 8, 1.0, SEED, 0)       # keep all
    kvc.kvc_random_evict(cache, 40, 0.5, SEED, 1)      # no candidates: no-op
    torch.cuda.synchronize()
    assert cache.n.cpu().eq(40).all() and torch.equal(cache.K, before)
    with pytest.raises(kvc.KvcError):
        kvc.kvc_random_evict(cache, 8, 1.5, SEED, 0)
