"""Paged slot-cache layout (block tables of 64-slot pages in a shared pool).

Every slot-cache operation runs on a dense cache and on a paged cache whose units own shuffled
pages of one pool; the paged run must give bit-identical logical contents (K, V, pos, n,
scores) and outputs -- the dense path is pinned to the oracle by the other test files.  A
ragged batch (units holding only the pages they need, -1 beyond) is checked against the oracle
directly, and a write through a missing page is skipped and flagged."""
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


def _gather(cache):
    """Logical [B, Hkv, C, D] K and V of a paged cache (through its block table)."""
    B, Hkv, C, D = cache.B, cache.Hkv, cache.C, cache.D
    tbl = cache.block_table.long().clamp(min=0)                     # [B, Hkv, C/64]
    rows = (tbl[..., :, None] * 64 + torch.arange(64, device=tbl.device)).reshape(B, Hkv, C)
    K = cache.K.reshape(-1, D)[rows.reshape(-1)].reshape(B, Hkv, C, D)
    V = cache.V.reshape(-1, D)[rows.reshape(-1)].reshape(B, Hkv, C, D)
    return K, V


def _assert_same(dense, paged, scores_d=None, scores_p=None):
    torch.cuda.synchronize()
    assert torch.equal(dense.n, paged.n) and torch.equal(dense.seqlen, paged.seqlen)
    Kp, Vp = _gather(paged)
    for b in range(dense.B):
        for h in range(dense.Hkv):
            nn = int(dense.n[b, h])
            assert torch.equal(dense.pos[b, h, :nn], paged.pos[b, h, :nn])
            assert torch.equal(dense.K[b, h, :nn], Kp[b, h, :nn]), (b, h)
            assert torch.equal(dense.V[b, h, :nn], Vp[b, h, :nn]), (b, h)
            if scores_d is not None:
                assert torch.equal(scores_d[b, h, :nn], scores_p[b, h, :nn])


def _attend(kvc, cache, q, logits=False, scores=None, decay=0.0):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda")
    lg = torch.empty(q.shape[0], q.shape[1], cache.C, dtype=torch.float32, device="cuda") \
        if logits else None
    splits = 1 if scores is not None else 0
    ws = torch.empty(max(kvc.kvc_workspace_size(cache, q, splits) // 4, 1), device="cuda")
    kvc.kvc_decode_attend(cache, q, o, logits=lg, lse=lse, workspace=ws, num_splits=splits,
                          h2o_scores=scores, h2o_decay=decay)
    return o, lse


def _pair(kvc, B, Hkv, C, D, spare=7, seed=0):
    """A dense cache and a paged twin whose units own shuffled pages of one pool."""
    dense = kvc.SlotCache.empty(B, Hkv, C, D)
    npu = C // 64
    num_pages = B * Hkv * npu + spare
    perm = torch.from_numpy(np.random.default_rng(seed).permutation(num_pages)[:B * Hkv * npu]
                            .astype(np.int32)).view(B, Hkv, npu)
    paged = kvc.SlotCache.empty_paged(B, Hkv, C, D, num_pages, block_table=perm)
    return dense, paged


@pytest.mark.parametrize("D", [128, 64])
def test_paged_equals_dense_through_every_method(kvc, D):
    B, Hq, Hkv, C, P, steps = 3, 16, 4, 704, 600, 6
    n_heavy, n_recent, n_sink = 40, 100, 16
    g = torch.Generator().manual_seed(D)
    Ks = torch.randn(B, Hkv, P + steps, D, generator=g).half().cuda()
    Vs = torch.randn(B, Hkv, P + steps, D, generator=g).half().cuda()
    qs = torch.randn(steps + 1, B, Hq, D, generator=g).half().cuda()
    prompt_k, prompt_v = Ks[:, :, :P].contiguous(), Vs[:, :, :P].contiguous()
    # FP16: bulk append of the prompt, then attention (automatic splits)
    dense, paged = _pair(kvc, B, Hkv, C, D, seed=D)
    for c in (dense, paged):
        kvc.kvc_append(c, prompt_k, prompt_v)
    _assert_same(dense, paged)
    od, ld = _attend(kvc, dense, qs[0])
    op, lp = _attend(kvc, paged, qs[0])
    assert torch.equal(od, op) and torch.equal(ld, lp)
    # H2O: seeded scores, evict to budget, then decode steps with the fused update and the
    # batched trigger; StreamingLLM and random eviction on twins of the same prompt
    rng = np.random.default_rng(D)
    sc0 = torch.from_numpy(rng.uniform(0, 4, (B, Hkv, C)).astype(np.float32)).cuda()
    sd, sp = sc0.clone(), sc0.clone()
    kvc.kvc_h2o_evict(dense, sd, n_heavy, n_recent)
    kvc.kvc_h2o_evict(paged, sp, n_heavy, n_recent)
    _assert_same(dense, paged, sd, sp)
    for t in range(steps):
        kn = Ks[:, :, P + t:P + t + 1].contiguous()
        vn = Vs[:, :, P + t:P + t + 1].contiguous()
        outs = []
        for c, s in ((dense, sd), (paged, sp)):
            kvc.kvc_append(c, kn, vn)
            outs.append(_attend(kvc, c, qs[t + 1], logits=True, scores=s, decay=0.99))
            kvc.kvc_h2o_evict_when(c, s, n_heavy, n_recent, n_heavy + n_recent + 3)
        assert torch.equal(outs[0][0], outs[1][0])
        _assert_same(dense, paged, sd, sp)
    for evict in ("stream", "random"):
        dense, paged = _pair(kvc, B, Hkv, C, D, seed=D + len(evict))
        for c in (dense, paged):
            kvc.kvc_append(c, prompt_k, prompt_v)
            if evict == "stream":
                kvc.kvc_stream_evict(c, n_sink, n_recent)
            else:
                kvc.kvc_random_evict(c, 64, 0.25, SEED, 0)
        _assert_same(dense, paged)
        od, _ = _attend(kvc, dense, qs[1])
        op, _ = _attend(kvc, paged, qs[1])
        assert torch.equal(od, op)
    assert device_status_clean(kvc)


def test_ragged_paged_batch_against_oracle(kvc, orc):
    """Units of one batch hold different token counts and only the pages those need (-1
    beyond); decode attention over them matches the oracle unit by unit."""
    B, Hq, Hkv, D, C = 2, 8, 4, 128, 1024
    counts = np.array([[1000, 65, 1, 640], [257, 0, 999, 64]], np.int32)
    g = torch.Generator().manual_seed(5)
    K = torch.randn(B, Hkv, C, D, generator=g).half()
    V = torch.randn(B, Hkv, C, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    need = (counts + 63) // 64
    num_pages = int(need.sum()) + 3
    order = np.random.default_rng(6).permutation(num_pages)
    table = np.full((B, Hkv, C // 64), -1, np.int32)
    k = 0
    for b in range(B):
        for h in range(Hkv):
            table[b, h, :need[b, h]] = order[k:k + need[b, h]]
            k += need[b, h]
    cache = kvc.SlotCache.empty_paged(B, Hkv, C, D, num_pages,
                                      block_table=torch.from_numpy(table))
    rows, src = [], []
    for b in range(B):
        for h in range(Hkv):
            j = np.arange(counts[b, h])
            rows.append(table[b, h, j // 64].astype(np.int64) * 64 + j % 64)
            src.append((b * Hkv + h) * C + j)
    rows = torch.from_numpy(np.concatenate(rows)).cuda()
    src = torch.from_numpy(np.concatenate(src)).cuda()
    cache.K.view(-1, D)[rows] = K.cuda().reshape(-1, D)[src]
    cache.V.view(-1, D)[rows] = V.cuda().reshape(-1, D)[src]
    cache.n.copy_(torch.from_numpy(counts).cuda())
    cache.seqlen.copy_(torch.from_numpy(counts.max(1)).cuda())
    for splits in (0, 1, 3):
        o = torch.empty(B, Hq, D, dtype=torch.float16, device="cuda")
        ws = torch.empty(max(kvc.kvc_workspace_size(cache, q.cuda(), splits) // 4, 1),
                         device="cuda")
        kvc.kvc_decode_attend(cache, q.cuda(), o, workspace=ws, num_splits=splits)
        ref, _, _ = orc.decode_attend(np16(q), np16(K), np16(V), counts)
        assert_o_close(np16(o), ref, what=f"splits={splits}")
    assert device_status_clean(kvc)


def test_write_through_a_missing_page_is_flagged(kvc):
    """A unit whose next slot has no page (-1 entry): the append skips the row and sets the
    capacity bit; nothing outside the pool is written."""
    B, Hkv, D, C = 1, 2, 128, 128
    table = torch.tensor([[[0, -1], [1, 2]]], dtype=torch.int32)
    cache = kvc.SlotCache.empty_paged(B, Hkv, C, D, 3, block_table=table)
    cache.n.fill_(64)                      # unit 0 is full up to its only page
    cache.seqlen.fill_(64)
    guard = cache.K.clone()
    k = torch.ones(B, Hkv, 1, D, dtype=torch.float16, device="cuda")
    kvc.kvc_append(cache, k, k)
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status() & kvc.KVC_DEV_CAPACITY
    # unit 1's slot 64 landed in its second page (pool page 2, row 0); unit 0 wrote nothing
    assert torch.equal(cache.K[2, 0], k[0, 1, 0])
    assert torch.equal(cache.K[0], guard[0]) and torch.equal(cache.K[1], guard[1])
    assert kvc.kvc_read_device_status() == 0


def _gather_kivi(cache, pools=("k_blocks", "v_blocks")):
    """Logical [B, Hkv, Cq/32, block] views of a paged KIVI cache's pools (the K and V blocks,
    or the GEAR side blocks)."""
    B, Hkv, Cq = cache.B, cache.Hkv, cache.Cq
    tbl = cache.block_table.long().clamp(min=0)                     # [B, Hkv, Cq/128]
    idx = (tbl[..., :, None] * 4 + torch.arange(4, device=tbl.device)).reshape(-1)
    out = []
    for name in pools:
        pool = getattr(cache, name)
        bb = pool.shape[-1]
        out.append(pool.reshape(-1, bb)[idx].reshape(B, Hkv, Cq // 32, bb))
    return tuple(out)


def _attend_kivi(kvc, cache, q, splits=0):
    o = torch.empty_like(q)
    ws = torch.empty(max(kvc.kvc_workspace_size(cache, q, splits) // 4, 1), device="cuda")
    kvc.kvc_decode_attend(cache, q, o, workspace=ws, num_splits=splits)
    return o


@pytest.mark.parametrize("D,bits,R,gear", [(128, 4, 128, False), (128, 2, 16, False),
                                            (64, 4, 32, False), (128, 4, 128, True),
                                            (64, 4, 32, True)])
def test_paged_kivi_equals_dense(kvc, D, bits, R, gear):
    """KIVI (and GEAR: side blocks in pools behind the same table) through shuffled pages:
    bulk and decode appends write the same blocks as the dense layout, and attention is
    bit-identical."""
    B, Hq, Hkv, P, steps, Cq = 3, 8, 2, 500, 40, 640
    g = torch.Generator().manual_seed(D + bits + R)
    Ks = torch.randn(B, Hkv, P + steps, D, generator=g).half().cuda()
    Vs = torch.randn(B, Hkv, P + steps, D, generator=g).half().cuda()
    q = torch.randn(B, Hq, D, generator=g).half().cuda()
    npu = Cq // 128
    num_pages = B * Hkv * npu + 5
    perm = torch.from_numpy(np.random.default_rng(D + bits).permutation(num_pages)
                            [:B * Hkv * npu].astype(np.int32)).view(B, Hkv, npu)
    dense = kvc.QuantCache.empty(B, Hkv, Cq, D, bits, R, gear=gear)
    paged = kvc.QuantCache.empty_paged(B, Hkv, Cq, D, bits, R, num_pages, block_table=perm,
                                       gear=gear)
    for c in (dense, paged):
        kvc.kvc_append_quant(c, Ks[:, :, :P].contiguous(), Vs[:, :, :P].contiguous())
    for t in range(steps + 1):
        if t > 0:
            for c in (dense, paged):
                kvc.kvc_append_quant(c, Ks[:, :, P + t - 1:P + t].contiguous(),
                                     Vs[:, :, P + t - 1:P + t].contiguous())
        if t % 8 == 0:
            torch.cuda.synchronize()
            kb, vb = _gather_kivi(paged)
            n_groups = (P + t - R) // 32 if P + t > R else 0
            assert torch.equal(dense.k_blocks[:, :, :n_groups], kb[:, :, :n_groups])
            assert torch.equal(dense.v_blocks[:, :, :n_groups], vb[:, :, :n_groups])
            assert torch.equal(dense.k_res, paged.k_res) and torch.equal(dense.v_res, paged.v_res)
            if gear:
                kg, vg = _gather_kivi(paged, ("k_gear", "v_gear"))
                assert torch.equal(dense.k_gear[:, :, :n_groups], kg[:, :, :n_groups])
                assert torch.equal(dense.v_gear[:, :, :n_groups], vg[:, :, :n_groups])
            for splits in (0, 2):
                assert torch.equal(_attend_kivi(kvc, dense, q, splits),
                                   _attend_kivi(kvc, paged, q, splits))
    assert device_status_clean(kvc)


def test_ragged_paged_kivi_against_oracle(kvc, orc):
    """Sequences of different lengths in one paged KIVI batch, each unit holding only the pages
    its quantised groups need (-1 beyond): blocks bit-exact and attention matches the oracle."""
    B, Hq, Hkv, D, bits, R, Cq = 3, 8, 2, 128, 4, 128, 1024
    lens = [1100, 130, 600]
    g = torch.Generator().manual_seed(77)
    T = max(lens)
    K = torch.randn(B, Hkv, T, D, generator=g).half()
    V = torch.randn(B, Hkv, T, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    n_q = [orc.kivi_nq(L, R) for L in lens]
    need = [(nq + 127) // 128 for nq in n_q]
    num_pages = Hkv * sum(need) + 2
    order = np.random.default_rng(78).permutation(num_pages)
    table = np.full((B, Hkv, Cq // 128), -1, np.int32)
    k = 0
    for b in range(B):
        for h in range(Hkv):
            table[b, h, :need[b]] = order[k:k + need[b]]
            k += need[b]
    cache = kvc.QuantCache.empty_paged(B, Hkv, Cq, D, bits, R, num_pages,
                                       block_table=torch.from_numpy(table))
    # each sequence gets its own length: append per sequence through one-sequence views
    for b in range(B):
        view = kvc.QuantCache(k_blocks=cache.k_blocks, v_blocks=cache.v_blocks,
                              k_res=cache.k_res[b:b + 1], v_res=cache.v_res[b:b + 1],
                              len=cache.len[b:b + 1], bits=bits, R=R,
                              block_table=cache.block_table[b:b + 1], Cq_paged=Cq)
        kvc.kvc_append_quant(view, K[b:b + 1, :, :lens[b]].cuda().contiguous(),
                             V[b:b + 1, :, :lens[b]].cuda().contiguous())
    torch.cuda.synchronize()
    kb, vb = _gather_kivi(cache)
    o = _attend_kivi(kvc, cache, q.cuda())
    gq = Hq // Hkv
    for b in range(B):
        for h in range(Hkv):
            Kb, Vb = np16(K[b, h, :lens[b]]), np16(V[b, h, :lens[b]])
            qz = orc.kivi_quantize_unit(Kb[:n_q[b]], Vb[:n_q[b]], n_q[b], bits)
            rk, rv = orc.kivi_pack_unit(qz, D, bits)
            ng = n_q[b] // 32
            assert np.array_equal(kb[b, h, :ng].cpu().numpy(), rk[:ng])
            assert np.array_equal(vb[b, h, :ng].cpu().numpy(), rv[:ng])
            ref, _ = orc.kivi_attend_unit(np16(q[b, h * gq:(h + 1) * gq]), Kb, Vb, lens[b], R,
                                          bits, qz=qz)
            assert_o_close(np16(o[b, h * gq:(h + 1) * gq]), ref, what=f"b={b} h={h}")
    assert device_status_clean(kvc)
