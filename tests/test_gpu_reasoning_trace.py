"""GPU parity over the whole reasoning-trace workload ("KV Cache 驱逐实战", section "参考实现":
per-head uniform random eviction with the prompt locked, applied every 1024 generated tokens).

Qwen3-32B-shaped layer: 16 sequences, GQA 64/8, head dim 128, a locked prompt of 1024 tokens,
the trace grown to 32768 tokens, 31 evictions to keep 0.25 of the generated tokens per KV head,
and decode attention after every eviction.  At every eviction:
  - every one of the 128 units keeps exactly the oracle's set (bit-exact positions), with the
    per-head count 1024 + 256, 320, 336, 340, 341, 341, ...;
  - every kept slot of every unit holds its token's original K and V rows (bit-exact);
  - attention of two sequences (all 64 query heads, rotating over the batch) is within the
    fp16 output tolerance of the fp64 oracle.
"""
import numpy as np
import pytest
import torch

from helpers import LSE_ABS_TOL, assert_o_close, device_status_clean, np16

pytestmark = pytest.mark.gpu
SEED = 0x243F6A8885A308D3


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def test_random_reasoning_full_trace(kvc, orc):
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.REASONING
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    P, every, T_end = w.prompt_len, w.evict_every, w.T
    n_evict = (T_end - P) // every
    assert n_evict == 31
    Kseq, Vseq = W.kv_tensors(w, T=T_end, device="cuda")
    C = 2432                                     # >= 1024 + 341 + 1024 slots before an eviction
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    kvc.kvc_append(cache, Kseq[:, :, :P + every].contiguous(), Vseq[:, :, :P + every].contiguous())
    o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    cur = {(b, h): np.arange(P + every, dtype=np.int32) for b in range(B) for h in range(Hkv)}
    counts = []
    for e in range(n_evict):
        if e > 0:
            t0 = P + every * e
            kvc.kvc_append(cache, Kseq[:, :, t0:t0 + every].contiguous(),
                           Vseq[:, :, t0:t0 + every].contiguous())
            for k in cur:
                cur[k] = np.concatenate([cur[k], np.arange(t0, t0 + every, dtype=np.int32)])
        kvc.kvc_random_evict(cache, P, w.keep_ratio, SEED, e)
        q = W.q_tensor(w, device="cuda", seed_offset=e)
        ws = torch.empty(max(kvc.kvc_workspace_size(cache, q) // 4, 1), dtype=torch.float32,
                         device="cuda")
        kvc.kvc_decode_attend(cache, q, o, lse=lse, workspace=ws)
        torch.cuda.synchronize()

        # keep-sets of all units against the oracle
        n = cache.n.cpu().numpy()
        pos = cache.pos.cpu().numpy()
        for (b, h), p in cur.items():
            keep = orc.random_keep(p, P, w.keep_ratio, SEED, e, b, h)
            cur[(b, h)] = p[keep]
        kept = len(cur[(0, 0)])
        counts.append(kept - P)
        assert (n == kept).all(), f"eviction {e}: counts {np.unique(n)} vs {kept}"
        for (b, h), p in cur.items():
            got = pos[b, h, :kept]
            assert np.array_equal(np.sort(got), p), f"eviction {e}: unit ({b},{h}) keep-set"
        # K / V rows of every kept slot, compared on the device
        idx = cache.pos[:, :, :kept].long()[..., None].expand(B, Hkv, kept, D)
        assert torch.equal(cache.K[:, :, :kept], torch.gather(Kseq, 2, idx)), f"eviction {e}: K"
        assert torch.equal(cache.V[:, :, :kept], torch.gather(Vseq, 2, idx)), f"eviction {e}: V"
        # attention of two sequences (all heads) against the oracle, over the kept tokens
        bs = [(2 * e) % B, (2 * e + 1) % B]
        Ks = np.stack([np.stack([np16(Kseq[b, h, torch.as_tensor(cur[(b, h)]).cuda().long()])
                                 for h in range(Hkv)]) for b in bs])
        Vs = np.stack([np.stack([np16(Vseq[b, h, torch.as_tensor(cur[(b, h)]).cuda().long()])
                                 for h in range(Hkv)]) for b in bs])
        ref, ref_lse, _ = orc.decode_attend(np16(q[bs]), Ks, Vs, np.full((2, Hkv), kept),
                                            threads=8)
        assert_o_close(np16(o[bs]).astype(np.float64), ref, what=f"eviction {e} o")
        assert np.abs(lse[bs].cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_ABS_TOL
    expect = [256, 320, 336, 340, 341] + [341] * (n_evict - 5)
    assert counts == expect
    assert device_status_clean(kvc)
