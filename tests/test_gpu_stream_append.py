"""GPU parity of the StreamingLLM decode append (kvc_stream_append): the token that leaves the
window gives up its slot to the new token, so no eviction launch runs in decode
("Rethinking KV Cache Compression" guide, §2 and §16 "4 种方法逐步执行": sinks plus the recent
window, no scores).  After every call a unit holds exactly this step's attention window,
positions < n_sink and P - n_recent .. P (the closed form of the oracle's stream_keep with a
window one token wider, evaluated at T = P + 1), each slot with its token's K and V rows, and
decode attention over it matches the fp64 oracle."""
import numpy as np
import pytest
import torch

from helpers import assert_o_close, device_status_clean, np16, slot_cache_from

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def _window(orc, T, n_sink, n_recent):
    """Positions of the attention window after appending token T - 1."""
    return np.flatnonzero(orc.stream_keep(np.arange(T), T, n_sink, n_recent + 1))


def test_stream_append_full_size_decode(kvc, orc):
    """The heavy-load StreamingLLM-512 decode at the benchmark's shape: 512 sequences, GQA 64/8,
    D 128, a 2047-token prompt gathered to 64 sinks + 448 recent, then 40 decode steps of
    kvc_stream_append + attention.  Every step: every unit's positions against the closed form,
    every kept row of every unit against its token (on the device), attention of two sequences
    against the oracle."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.HEAVY
    B, Hq, Hkv, D, n_sink, n_recent = w.B, w.Hq, w.Hkv, w.D, w.n_sink, w.n_recent
    L, steps, C = w.T - 1, 40, 520
    Kseq, Vseq = W.kv_tensors(w, T=L + steps, B=B, device="cuda")
    full = kvc.SlotCache.empty(B, Hkv, L + 8, D)
    kvc.kvc_append(full, Kseq[:, :, :L].contiguous(), Vseq[:, :, :L].contiguous())
    kvc.kvc_stream_evict(full, n_sink, n_recent)
    cache = kvc.SlotCache.empty(B, Hkv, C, D)
    cache.K[:, :, :512] = full.K[:, :, :512]
    cache.V[:, :, :512] = full.V[:, :, :512]
    cache.pos[:, :, :512] = full.pos[:, :, :512]
    cache.n.copy_(full.n)
    cache.seqlen.copy_(full.seqlen)
    del full
    o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    for s in range(steps):
        P = L + s
        kvc.kvc_stream_append(cache, Kseq[:, :, P:P + 1].contiguous(),
                              Vseq[:, :, P:P + 1].contiguous(), n_sink, n_recent)
        q = W.q_tensor(w, device="cuda", seed_offset=s)
        ws = torch.empty(max(kvc.kvc_workspace_size(cache, q) // 4, 1), dtype=torch.float32,
                         device="cuda")
        kvc.kvc_decode_attend(cache, q, o, workspace=ws)
        torch.cuda.synchronize()
        want = _window(orc, P + 1, n_sink, n_recent)
        n = cache.n.cpu().numpy()
        assert (n == len(want)).all() and len(want) == 513, f"step {s}"
        assert (cache.seqlen.cpu().numpy() == P + 1).all()
        got = np.sort(cache.pos[:, :, :513].cpu().numpy(), axis=2)
        assert (got == want[None, None, :]).all(), f"step {s}: window"
        idx = cache.pos[:, :, :513].long()[..., None].expand(B, Hkv, 513, D)
        assert torch.equal(cache.K[:, :, :513], torch.gather(Kseq, 2, idx)), f"step {s}: K"
        assert torch.equal(cache.V[:, :, :513], torch.gather(Vseq, 2, idx)), f"step {s}: V"
        bs = [(37 * s) % B, (37 * s + 11) % B]
        wi = torch.as_tensor(want).long().cuda()
        ref, _, _ = orc.decode_attend(np16(q[bs]), np16(Kseq[bs][:, :, wi]),
                                      np16(Vseq[bs][:, :, wi]), np.full((2, Hkv), 513),
                                      threads=8)
        assert_o_close(np16(o[bs]).astype(np.float64), ref, what=f"step {s} o")
    assert device_status_clean(kvc)


@pytest.mark.parametrize("T0,n_sink,n_recent,steps,paged", [
    (1, 4, 12, 40, False),       # window fills up during the run, then slides
    (20, 0, 8, 30, False),       # no sinks
    (70, 4, 12, 24, True),       # paged twin of a sliding window
    (5, 16, 4, 40, False),       # sinks larger than the recent window
])
def test_stream_append_small_windows(kvc, orc, T0, n_sink, n_recent, steps, paged):
    """Tiny workload shapes (MHA 4 heads, D 64): the prompt gathered by kvc_stream_evict (or
    short enough to need none), then decode steps; the window grows until it holds
    n_sink + n_recent + 1 tokens and then slides with n fixed."""
    B, Hq, Hkv, D = 2, 4, 4, 64
    C = 128
    g = torch.Generator().manual_seed(T0 * 7 + n_recent)
    Kseq = torch.randn(B, Hkv, T0 + steps, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, T0 + steps, D, generator=g).half()
    q_all = torch.randn(steps, B, Hq, D, generator=g).half()
    if paged:
        npu = C // 64
        table = torch.randperm(B * Hkv * npu, generator=g).int().view(B, Hkv, npu).cuda()
        cache = kvc.SlotCache.empty_paged(B, Hkv, C, D, B * Hkv * npu, block_table=table)
        cache.seqlen.zero_()
        cache.n.zero_()
        kvc.kvc_append(cache, Kseq[:, :, :T0].cuda().contiguous(), Vseq[:, :, :T0].cuda().contiguous())
    else:
        cache = slot_cache_from(kvc, Kseq[:, :, :T0], Vseq[:, :, :T0], np.full((B, Hkv), T0), C,
                                seqlen=[T0] * B)
    kvc.kvc_stream_evict(cache, n_sink, n_recent)
    o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
    for s in range(steps):
        P = T0 + s
        kvc.kvc_stream_append(cache, Kseq[:, :, P:P + 1].cuda().contiguous(),
                              Vseq[:, :, P:P + 1].cuda().contiguous(), n_sink, n_recent)
        q = q_all[s].cuda()
        ws = torch.empty(max(kvc.kvc_workspace_size(cache, q) // 4, 1), dtype=torch.float32,
                         device="cuda")
        kvc.kvc_decode_attend(cache, q, o, workspace=ws)
        torch.cuda.synchronize()
        want = _window(orc, P + 1, n_sink, n_recent)
        n = cache.n.cpu().numpy()
        assert (n == len(want)).all(), f"step {s}: n {np.unique(n)} vs {len(want)}"
        pos = cache.pos.cpu().numpy()
        Kg, Vg = cache.K.cpu(), cache.V.cpu()
        for b in range(B):
            for h in range(Hkv):
                got = pos[b, h, :len(want)]
                assert np.array_equal(np.sort(got), want), f"step {s} unit ({b},{h})"
                if paged:
                    tab = table.cpu().numpy()
                    rows = [tab[b, h, j // 64] * 64 + j % 64 for j in range(len(want))]
                    kr, vr = Kg.view(-1, D)[rows], Vg.view(-1, D)[rows]
                else:
                    kr, vr = Kg[b, h, :len(want)], Vg[b, h, :len(want)]
                gi = torch.as_tensor(got).long()
                assert torch.equal(kr, Kseq[b, h, gi]) and torch.equal(vr, Vseq[b, h, gi])
        wi = torch.as_tensor(want).long()
        ref, _, _ = orc.decode_attend(np16(q), np16(Kseq[:, :, wi]), np16(Vseq[:, :, wi]),
                                      np.full((B, Hkv), len(want)))
        assert_o_close(np16(o).astype(np.float64), ref, what=f"step {s} o")
    assert device_status_clean(kvc)


def test_stream_append_capacity_flag(kvc):
    """A unit whose window is still growing and whose cache is full is left unchanged and
    flags KVC_DEV_CAPACITY; the sequence length still advances."""
    B, Hkv, D, C = 1, 2, 64, 16
    g = torch.Generator().manual_seed(16)
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    cache = slot_cache_from(kvc, K, K, np.full((B, Hkv), C), C, seqlen=[C])
    kn = torch.randn(B, Hkv, 1, D, generator=g).half().cuda()
    before = cache.K.clone()
    kvc.kvc_stream_append(cache, kn, kn, 4, 100)   # window not full: the token needs slot C
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status() & kvc.KVC_DEV_CAPACITY
    assert cache.n.cpu().eq(C).all() and torch.equal(cache.K, before)
    with pytest.raises(ValueError):
        kvc.kvc_stream_append(cache, torch.zeros(B, Hkv, 2, D, dtype=torch.float16, device="cuda"),
                              torch.zeros(B, Hkv, 2, D, dtype=torch.float16, device="cuda"), 4, 8)
