"""GPU parity of the LLaMA-7B-shaped H2O-512 path as the pages run it ("Rethinking KV Cache
Compression" guide, §2: 64 heavy + 448 recent; §16 "4 种方法逐步执行" and "局限与最终结论": prompt
scores from an extra pass over the causal prompt, then accumulate and update the keep set at
every decode step).

8 sequences, 32 MHA heads, head dim 128, K and V with 2% outlier channels scaled x10 per KV
head; a 2048-token causal prompt with queries ~ N(0,1):
  1. the two-pass prefill score pass over the whole batch -- every unit's scores sum to L
     (conservation), sampled units against the oracle within 1e-4 relative;
  2. eviction 2048 -> 512 -- sampled units' keep-sets against the oracle's (near-ties within
     1e-6 relative may swap), every unit's rows against its tokens;
  3. one decode step in the benchmark's launch: append token 2048, attention over the 513 slots
     with the score update fused (logits on chip), eviction 513 -> 512 -- sampled units' o, lse,
     scores and keep-sets against the oracle run from its own post-prefill state (its keep-set
     and prefill scores; a unit whose keep-set differs by an accepted near-tie is skipped).
"""
import numpy as np
import pytest
import torch

from helpers import (LSE_ABS_TOL, SCORE_REL_TOL, assert_o_close, device_status_clean, np16)
from test_gpu_evict import _check_keep_with_ties

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def test_llama7b_h2o512_prefill_evict_and_decode(kvc, orc):
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.LLAMA7B
    B, Hq, Hkv, D, L = w.B, w.Hq, w.Hkv, w.D, w.T
    n_heavy, n_recent = w.n_heavy, w.n_recent
    K, V = W.kv_tensors(w, T=L + 1, device="cuda")
    qp = W.q_tensor(w, L=L, device="cuda")
    q = W.q_tensor(w, device="cuda", seed_offset=1)
    C0 = L + 8
    full = kvc.SlotCache.empty(B, Hkv, C0, D)
    kvc.kvc_append(full, K[:, :, :L].contiguous(), V[:, :, :L].contiguous())
    scores0 = torch.zeros(B, Hkv, C0, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvc.kvc_h2o_workspace_size(B, Hq, L) // 4, dtype=torch.float32,
                     device="cuda")
    kvc.kvc_h2o_accumulate_prefill(qp, full.K, scores0, ws, L)
    torch.cuda.synchronize()
    assert device_status_clean(kvc)
    tot = scores0[..., :L].double().sum(dim=2).cpu().numpy()
    np.testing.assert_allclose(tot, float(L), rtol=1e-4)      # g = 1: each row sums to 1
    prefill_scores = scores0[..., :L].cpu().numpy().astype(np.float64)

    rng = np.random.default_rng(2048)
    units = sorted({(0, 0), (B - 1, Hkv - 1)} |
                   {(int(b), int(h)) for b, h in zip(rng.integers(0, B, 3), rng.integers(0, Hkv, 3))})
    ref_pre = {}
    for b, h in units:
        ref = orc.h2o_prefill_scores(np16(qp[b:b + 1, h:h + 1]), np16(K[b:b + 1, h:h + 1, :L]), L,
                                     threads=8)[0, 0]
        np.testing.assert_allclose(prefill_scores[b, h], ref, rtol=SCORE_REL_TOL, atol=0,
                                   err_msg=f"prefill scores ({b},{h})")
        ref_pre[(b, h)] = ref

    # 2. eviction of the prompt to 64 heavy + 448 recent
    kvc.kvc_h2o_evict(full, scores0, n_heavy, n_recent)
    torch.cuda.synchronize()
    assert (full.n.cpu().numpy() == 512).all()
    for b, h in units:
        _check_keep_with_ties(full.pos[b, h, :512].cpu().numpy(), np.arange(L, dtype=np.int32),
                              ref_pre[(b, h)], L, n_heavy, n_recent)
    idx = full.pos[:, :, :512].long()[..., None].expand(B, Hkv, 512, D)
    assert torch.equal(full.K[:, :, :512], torch.gather(K, 2, idx))
    assert torch.equal(full.V[:, :, :512], torch.gather(V, 2, idx))

    # 3. the decode step, in a 520-slot cache as the benchmark holds it
    C = 520
    c = kvc.SlotCache.empty(B, Hkv, C, D)
    c.K[:, :, :512] = full.K[:, :, :512]
    c.V[:, :, :512] = full.V[:, :, :512]
    c.pos[:, :, :512] = full.pos[:, :, :512]
    c.n.copy_(full.n)
    c.seqlen.copy_(full.seqlen)
    sc = torch.zeros(B, Hkv, C, dtype=torch.float32, device="cuda")
    sc[:, :, :512] = scores0[:, :, :512]
    pos512 = c.pos[:, :, :512].cpu().numpy()
    del full, scores0
    o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    kvc.kvc_append(c, K[:, :, L:L + 1].contiguous(), V[:, :, L:L + 1].contiguous())
    kvc.kvc_decode_attend(c, q, o, lse=lse, h2o_scores=sc)
    sc_mid = sc.clone()
    kvc.kvc_h2o_evict(c, sc, n_heavy, n_recent)
    torch.cuda.synchronize()
    assert device_status_clean(kvc)
    assert (c.n.cpu().numpy() == 512).all()
    # the oracle's own state after its prefill eviction: its keep-set and prefill scores
    compared = 0
    for b, h in units:
        keep_ref, _ = orc.h2o_keep(np.arange(L, dtype=np.int32), ref_pre[(b, h)], L, n_heavy,
                                   n_recent)
        p_ref = np.flatnonzero(keep_ref).astype(np.int32)
        if set(p_ref.tolist()) != set(pos512[b, h].tolist()):
            continue   # a near-tie swap (accepted above): the two states differ by design
        compared += 1
        p = np.concatenate([p_ref, [L]]).astype(np.int32)
        pi = torch.from_numpy(p).long().cuda()
        ref_o, ref_lse, ref_lg = orc.decode_attend(np16(q[b:b + 1, h:h + 1]),
                                                   np16(K[b:b + 1, h:h + 1, pi]),
                                                   np16(V[b:b + 1, h:h + 1, pi]),
                                                   np.array([[513]], np.int32), want_logits=True)
        assert_o_close(np16(o[b:b + 1, h:h + 1]).astype(np.float64), ref_o, what=f"o ({b},{h})")
        assert abs(float(lse[b, h]) - ref_lse[0, 0]) <= LSE_ABS_TOL
        prev = np.concatenate([ref_pre[(b, h)][p_ref], [0.0]])[None, None]
        ref_sc = orc.h2o_accumulate(prev, ref_lg, ref_lse, np.array([[513]], np.int32))[0, 0]
        # the GPU's slots hold the prompt slots in its own order, then token L
        got = dict(zip(np.concatenate([pos512[b, h], [L]]).tolist(),
                       sc_mid[b, h, :513].cpu().numpy().astype(np.float64).tolist()))
        np.testing.assert_allclose([got[int(x)] for x in p], ref_sc, rtol=SCORE_REL_TOL,
                                   err_msg=f"scores ({b},{h})")
        _check_keep_with_ties(c.pos[b, h, :512].cpu().numpy(), p, ref_sc, L + 1, n_heavy,
                              n_recent)
    assert compared >= len(units) - 1
    idx = c.pos[:, :, :512].long()[..., None].expand(B, Hkv, 512, D)
    assert torch.equal(c.K[:, :, :512], torch.gather(K, 2, idx))
    assert torch.equal(c.V[:, :, :512], torch.gather(V, 2, idx))
