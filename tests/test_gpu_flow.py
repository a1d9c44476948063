"""GPU parity over a whole sequence of the tiny workload: a 64-token prompt, then 32 decode
steps of every method, each step's output compared with the fp64 oracle run free alongside.

Methods: full FP16; StreamingLLM (4 sinks + 12 recent); H2O (8 heavy + 8 recent, prefill
scores from the prompt queries); KIVI-4 (G=32, R=16); random eviction (keep 0.5, first 16
tokens locked) after the prompt and again after step 32.  Step order: append, attend over the
cache plus the new token, (H2O) add the probabilities, evict back to budget."""
import numpy as np
import pytest
import torch

from helpers import assert_o_close, device_status_clean, np16

pytestmark = pytest.mark.gpu
SEED = 0x243F6A8885A308D3


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


@pytest.fixture(scope="module")
def data():
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.TINY
    P, S = w.extra["prompt"], w.decode_steps
    K, V = W.kv_tensors(w, T=P + S)                  # [1, 4, 96, 64]
    Qp = W.q_tensor(w, L=P)                          # prompt queries [1, 4, 64, 64]
    qs = torch.stack([W.q_tensor(w, seed_offset=1 + t) for t in range(S)])   # [S, 1, 4, 64]
    return w, P, S, K, V, Qp, qs


def _attend(kvc, cache, q, logits=False):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda")
    lg = torch.empty(q.shape[0], q.shape[1], cache.C, dtype=torch.float32, device="cuda") \
        if logits else None
    ws = torch.empty(max(kvc.kvc_workspace_size(cache, q) // 4, 1), device="cuda")
    kvc.kvc_decode_attend(cache, q, o, logits=lg, lse=lse, workspace=ws)
    return o, lse, lg


def _orc_attend(orc, q, K, V, keep_pos, want_logits=False):
    """Oracle attention of q [1,Hq,D] over the positions keep_pos[h] of each KV head."""
    Hkv = K.shape[1]
    n = max(len(p) for p in keep_pos)
    Kc = np.zeros((1, Hkv, n, K.shape[-1]), np.float16)
    Vc = np.zeros_like(Kc)
    for h in range(Hkv):
        Kc[0, h, :len(keep_pos[h])] = K[0, h, keep_pos[h]]
        Vc[0, h, :len(keep_pos[h])] = V[0, h, keep_pos[h]]
    nn = np.array([[len(p) for p in keep_pos]], np.int32)
    return orc.decode_attend(q, Kc, Vc, nn, want_logits=want_logits)


def test_fp16_stream_kivi_sequence(kvc, orc, data):
    w, P, S, K, V, Qp, qs = data
    K16, V16 = np16(K), np16(V)
    Kc, Vc = K.cuda(), V.cuda()
    fp = kvc.SlotCache.empty(1, w.Hkv, 128, w.D)
    st = kvc.SlotCache.empty(1, w.Hkv, 32, w.D)
    kq = kvc.QuantCache.empty(1, w.Hkv, 128, w.D, 4, w.kivi_R)
    kvc.kvc_append(fp, Kc[:, :, :P].contiguous(), Vc[:, :, :P].contiguous())
    tmp = kvc.SlotCache.empty(1, w.Hkv, 96, w.D)
    kvc.kvc_append(tmp, Kc[:, :, :P].contiguous(), Vc[:, :, :P].contiguous())
    kvc.kvc_stream_evict(tmp, w.n_sink, w.n_recent)
    torch.cuda.synchronize()
    nst = int(tmp.n[0, 0])
    for name in ("K", "V", "pos"):
        getattr(st, name)[:, :, :nst] = getattr(tmp, name)[:, :, :nst]
    st.n.copy_(tmp.n)
    st.seqlen.copy_(tmp.seqlen)
    kvc.kvc_append_quant(kq, Kc[:, :, :P].contiguous(), Vc[:, :, :P].contiguous())
    g = w.Hq // w.Hkv
    for t in range(S):
        T = P + t + 1
        q = qs[t].cuda()
        kn, vn = Kc[:, :, T - 1:T].contiguous(), Vc[:, :, T - 1:T].contiguous()
        # FP16
        kvc.kvc_append(fp, kn, vn)
        o, _, _ = _attend(kvc, fp, q)
        ref, _, _ = orc.decode_attend(np16(q), K16[:, :, :T], V16[:, :, :T], np.full((1, w.Hkv), T))
        assert_o_close(np16(o), ref, what=f"fp16 step {t}")
        # StreamingLLM: the kept window of the previous length plus the new token
        kvc.kvc_append(st, kn, vn)
        o, _, _ = _attend(kvc, st, q)
        kept = np.flatnonzero(orc.stream_keep(np.arange(T - 1), T - 1, w.n_sink, w.n_recent))
        keep_pos = [np.concatenate([kept, [T - 1]])] * w.Hkv
        ref, _, _ = _orc_attend(orc, np16(q), K16, V16, keep_pos)
        assert_o_close(np16(o), ref, what=f"stream step {t}")
        kvc.kvc_stream_evict(st, w.n_sink, w.n_recent)
        # KIVI-4
        kvc.kvc_append_quant(kq, kn, vn)
        o, _, _ = _attend(kvc, kq, q)
        for h in range(w.Hkv):
            ref, _ = orc.kivi_attend_unit(np16(q[0, h * g:(h + 1) * g]), K16[0, h], V16[0, h], T,
                                          w.kivi_R, 4)
            assert_o_close(np16(o[0, h * g:(h + 1) * g]), ref, what=f"kivi step {t} head {h}")
    assert device_status_clean(kvc)


def test_h2o_sequence(kvc, orc, data):
    w, P, S, K, V, Qp, qs = data
    n_heavy, n_recent = w.n_heavy, w.extra["h2o_recent"]
    K16, V16 = np16(K), np16(V)
    Kc, Vc = K.cuda(), V.cuda()
    C = 64 + 8
    cache = kvc.SlotCache.empty(1, w.Hkv, C, w.D)
    kvc.kvc_append(cache, Kc[:, :, :P].contiguous(), Vc[:, :, :P].contiguous())
    scores = torch.zeros(1, w.Hkv, C, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvc.kvc_h2o_workspace_size(1, w.Hq, P) // 4, device="cuda")
    kvc.kvc_h2o_accumulate_prefill(Qp.cuda(), cache.K, scores, ws, P)
    kvc.kvc_h2o_evict(cache, scores, n_heavy, n_recent)
    torch.cuda.synchronize()
    # oracle prefill and keep-set
    ref_sc = orc.h2o_prefill_scores(np16(Qp), K16[:, :, :P].copy(), P)
    keep_pos, keep_sc = [], []
    for h in range(w.Hkv):
        k, _ = orc.h2o_keep(np.arange(P, dtype=np.int32), ref_sc[0, h], P, n_heavy, n_recent)
        keep_pos.append(np.flatnonzero(k))
        keep_sc.append(ref_sc[0, h][k])

    def gpu_state(h):
        nn = int(cache.n[0, h])
        return cache.pos[0, h, :nn].cpu().numpy(), scores[0, h, :nn].cpu().numpy()

    for h in range(w.Hkv):
        gp, _ = gpu_state(h)
        assert sorted(gp.tolist()) == sorted(keep_pos[h].tolist())
    g = w.Hq // w.Hkv
    for t in range(S):
        T = P + t + 1
        q = qs[t].cuda()
        kvc.kvc_append(cache, Kc[:, :, T - 1:T].contiguous(), Vc[:, :, T - 1:T].contiguous())
        o, lse, lg = _attend(kvc, cache, q, logits=True)
        kvc.kvc_h2o_accumulate_decode(cache, scores, lg, lse, w.Hq)
        kvc.kvc_h2o_evict(cache, scores, n_heavy, n_recent)
        torch.cuda.synchronize()
        step_pos = [np.concatenate([keep_pos[h], [T - 1]]) for h in range(w.Hkv)]
        ref, ref_lse, ref_lg = _orc_attend(orc, np16(q), K16, V16, step_pos, want_logits=True)
        assert_o_close(np16(o), ref, what=f"h2o step {t}")
        flipped = False
        for h in range(w.Hkv):
            n = len(step_pos[h])
            sc = np.concatenate([keep_sc[h], [0.0]])
            for hh in range(g):
                hq = h * g + hh
                sc += np.exp(ref_lg[0, hq, :n] - ref_lse[0, hq])
            k, margin = orc.h2o_keep(step_pos[h].astype(np.int32), sc, T, n_heavy, n_recent)
            keep_pos[h], keep_sc[h] = step_pos[h][k], sc[k]
            gp, gs = gpu_state(h)
            if sorted(gp.tolist()) != sorted(keep_pos[h].tolist()):
                # allowed only where the oracle's scores tie within 1e-6 relative
                assert margin <= 1e-6, (t, h, margin)
                flipped = True
            else:
                order = np.argsort(gp)
                np.testing.assert_allclose(gs[order], keep_sc[h][np.argsort(keep_pos[h])],
                                           rtol=1e-4)
        if flipped:
            break    # the runs legitimately diverge after a tie
    assert device_status_clean(kvc)


def test_random_sequence(kvc, orc, data):
    w, P, S, K, V, Qp, qs = data
    K16, V16 = np16(K), np16(V)
    Kc, Vc = K.cuda(), V.cuda()
    cache = kvc.SlotCache.empty(1, w.Hkv, 96, w.D)
    kvc.kvc_append(cache, Kc[:, :, :P].contiguous(), Vc[:, :, :P].contiguous())
    kvc.kvc_random_evict(cache, w.prompt_len, w.keep_ratio, SEED, 0)
    keep_pos = []
    for h in range(w.Hkv):
        k = orc.random_keep(np.arange(P, dtype=np.int32), w.prompt_len, w.keep_ratio, SEED, 0, 0, h)
        keep_pos.append(np.flatnonzero(k))
        assert len(keep_pos[h]) == 16 + 24
    for t in range(S):
        T = P + t + 1
        q = qs[t].cuda()
        kvc.kvc_append(cache, Kc[:, :, T - 1:T].contiguous(), Vc[:, :, T - 1:T].contiguous())
        o, _, _ = _attend(kvc, cache, q)
        keep_pos = [np.concatenate([p, [T - 1]]) for p in keep_pos]
        ref, _, _ = _orc_attend(orc, np16(q), K16, V16, keep_pos)
        assert_o_close(np16(o), ref, what=f"random step {t}")
    kvc.kvc_random_evict(cache, w.prompt_len, w.keep_ratio, SEED, 1)
    torch.cuda.synchronize()
    for h in range(w.Hkv):
        p = keep_pos[h].astype(np.int32)
        k = orc.random_keep(p, w.prompt_len, w.keep_ratio, SEED, 1, 0, h)
        nn = int(cache.n[0, h])
        assert nn == 16 + 28
        assert sorted(cache.pos[0, h, :nn].cpu().tolist()) == sorted(p[k].tolist())
    assert device_status_clean(kvc)
