"""GPU parity: KIVI packing (bit-exact vs the oracle) and KIVI decode attention."""
import numpy as np
import pytest
import torch

from helpers import assert_o_close, device_status_clean, np16

pytestmark = pytest.mark.gpu
G = 32
# The per-channel K scale is folded into the query, q~ = q * s rounded to binary16 (relative
# error <= 2^-12 per product), so a KIVI logit carries up to ~1e-3 absolute error on these
# inputs; the outputs still meet the 2e-3 bound, which assert_o_close checks.
KIVI_LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def _build(kvc, Kseq, Vseq, bits, R, Cq, chunks, offsets=None):
    """Append Kseq/Vseq [B,Hkv,T,D] through kvc_append_quant in the given chunk sizes.
    offsets[b] tokens of sequence b are pre-placed in the residual ring first (ragged lengths)."""
    B, Hkv, T, D = Kseq.shape
    cache = kvc.QuantCache.empty(B, Hkv, Cq, D, bits, R)
    off = np.zeros(B, np.int64) if offsets is None else np.asarray(offsets)
    for b in range(B):
        for p in range(off[b]):
            cache.k_res[b, :, p % (R + G)] = Kseq[b, :, p]
            cache.v_res[b, :, p % (R + G)] = Vseq[b, :, p]
    cache.len.copy_(torch.as_tensor(off, dtype=torch.int32))
    # per sequence b the appended stream is Kseq[b, :, off[b]:]
    t = 0
    for n_new in chunks:
        kn = torch.stack([Kseq[b, :, off[b] + t: off[b] + t + n_new] for b in range(B)]).contiguous()
        vn = torch.stack([Vseq[b, :, off[b] + t: off[b] + t + n_new] for b in range(B)]).contiguous()
        kvc.kvc_append_quant(cache, kn, vn)
        t += n_new
    torch.cuda.synchronize()
    return cache, off + t


def _check_unit(orc, cache, Kseq, Vseq, b, hk, T, bits, R):
    D = Kseq.shape[-1]
    n_q = orc.kivi_nq(T, R)
    Kb = np16(Kseq[b, hk, :T])
    Vb = np16(Vseq[b, hk, :T])
    if n_q > 0:
        qz = orc.kivi_quantize_unit(Kb[:n_q], Vb[:n_q], n_q, bits)
        kb, vb = orc.kivi_pack_unit(qz, D, bits)
        gk = cache.k_blocks[b, hk, :n_q // G].cpu().numpy()
        gv = cache.v_blocks[b, hk, :n_q // G].cpu().numpy()
        assert np.array_equal(gk, kb), f"K blocks differ at unit ({b},{hk})"
        assert np.array_equal(gv, vb), f"V blocks differ at unit ({b},{hk})"
    kr = cache.k_res[b, hk].cpu().numpy().view(np.uint16)
    vr = cache.v_res[b, hk].cpu().numpy().view(np.uint16)
    for p in range(n_q, T):
        s = p % (R + G)
        assert np.array_equal(kr[s], Kb[p].view(np.uint16)) and np.array_equal(vr[s], Vb[p].view(np.uint16))


@pytest.mark.parametrize("D,bits,R", [(128, 4, 128), (128, 2, 128), (64, 4, 16), (64, 2, 0),
                                      (128, 4, 100)])
def test_pack_bit_exact_with_flushes(kvc, orc, D, bits, R):
    g = torch.Generator().manual_seed(D + bits + R)
    B, Hkv = 3, 2
    chunks = [70] + [1] * 45 + [129, 3]
    offsets = [0, 5, min(R + G - 1, 37)]
    T = max(offsets) + sum(chunks)
    Kseq = (torch.randn(B, Hkv, T, D, generator=g) + torch.rand(1, Hkv, 1, D, generator=g) * 4 - 2).half()
    Vseq = (torch.randn(B, Hkv, T, D, generator=g) * 3).half()
    Kseq[0, 0, 32:64, 7] = 0.5         # a constant channel in one group -> scale 0
    Vseq[1, 1, 40, :] = -0.0           # a zero token -> zero stored as +0
    cache, lens = _build(kvc, Kseq.cuda(), Vseq.cuda(), bits, R, Cq=512, chunks=chunks,
                         offsets=offsets)
    assert cache.len.cpu().tolist() == list(lens)
    for b in range(B):
        for hk in range(Hkv):
            _check_unit(orc, cache, Kseq, Vseq, b, hk, int(lens[b]), bits, R)
    assert device_status_clean(kvc)


def test_decode_appends_over_more_units_than_one_wave(kvc, orc):
    """Decode-sized appends run one wave of CTAs that walk the units (six per SM); with 1280
    units every CTA takes more than one.  Sequences start at ragged lengths, so their groups
    flush at different steps; sampled units are checked bit-exactly."""
    B, Hkv, D, bits, R = 160, 8, 128, 4, 16
    g = torch.Generator().manual_seed(1280)
    offsets = [b % (R + G) for b in range(B)]
    chunks = [1] * 40
    T = max(offsets) + sum(chunks)
    Kseq = torch.randn(B, Hkv, T, D, generator=g).half()
    Vseq = torch.randn(B, Hkv, T, D, generator=g).half()
    assert B * Hkv > 6 * torch.cuda.get_device_properties(0).multi_processor_count
    cache, lens = _build(kvc, Kseq.cuda(), Vseq.cuda(), bits, R, Cq=128, chunks=chunks,
                         offsets=offsets)
    assert cache.len.cpu().tolist() == list(lens)
    rng = np.random.default_rng(3)
    for b in sorted({0, 1, 31, 47, 100, B - 1} | set(rng.integers(0, B, 4).tolist())):
        for hk in (0, int(rng.integers(0, Hkv)), Hkv - 1):
            _check_unit(orc, cache, Kseq, Vseq, b, hk, int(lens[b]), bits, R)
    assert device_status_clean(kvc)


def _attend(kvc, cache, q, splits=0):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda")
    ws = torch.empty(max(kvc.kvc_workspace_size(cache, q, splits) // 4, 1), dtype=torch.float32,
                     device="cuda")
    kvc.kvc_decode_attend(cache, q, o, lse=lse, workspace=ws, num_splits=splits)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("D,bits,R,Hq,Hkv,splits", [
    (64, 4, 16, 4, 4, 0), (128, 4, 128, 8, 1, 0), (128, 2, 128, 16, 2, 0), (64, 2, 0, 4, 2, 0),
    (128, 4, 100, 3, 3, 0), (128, 4, 128, 8, 2, 1), (128, 2, 16, 8, 2, 3), (64, 4, 16, 8, 1, 2)])
def test_attention_small(kvc, orc, D, bits, R, Hq, Hkv, splits):
    g = torch.Generator().manual_seed(7 * D + bits + Hq)
    B = 3
    chunks = [150, 1, 1, 33]
    offsets = [0, 9, 30]
    T = max(offsets) + sum(chunks)
    Kseq = (torch.randn(B, Hkv, T, D, generator=g) + torch.rand(1, Hkv, 1, D, generator=g) * 4 - 2).half()
    Vseq = (torch.randn(B, Hkv, T, D, generator=g) + torch.rand(1, Hkv, 1, D, generator=g) * 4 - 2).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    cache, lens = _build(kvc, Kseq.cuda(), Vseq.cuda(), bits, R, Cq=256, chunks=chunks,
                         offsets=offsets)
    o, lse = _attend(kvc, cache, q.cuda(), splits)
    gq = Hq // Hkv
    for b in range(B):
        for hk in range(Hkv):
            T_b = int(lens[b])
            ref, ref_lse = orc.kivi_attend_unit(np16(q[b, hk * gq:(hk + 1) * gq]),
                                                np16(Kseq[b, hk]), np16(Vseq[b, hk]), T_b, R, bits)
            assert_o_close(np16(o[b, hk * gq:(hk + 1) * gq]), ref, what=f"b={b} hk={hk}")
            np.testing.assert_allclose(lse[b, hk * gq:(hk + 1) * gq].cpu().numpy(), ref_lse,
                                       atol=KIVI_LSE_TOL, rtol=0)
    assert device_status_clean(kvc)


@pytest.mark.parametrize("wname,bits", [("kivi-b32-h32-d128-t4096", 2),
                                        ("kivi-b32-h32-d128-t4096", 4),
                                        ("heavy-gqa64x8-b512-d128-t2048", 4)])
def test_full_size_sampled(kvc, orc, wname, bits):
    """Full-size caches built by one bulk append (the prompt) and one decode append; sampled
    units are checked bit-exactly (blocks, ring) and for attention."""
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.WORKLOADS[wname]
    K, V = W.kv_tensors(w, device="cuda")
    q = W.q_tensor(w, device="cuda")
    Cq = orc.kivi_nq(w.T, w.kivi_R)
    cache = kvc.QuantCache.empty(w.B, w.Hkv, Cq, w.D, bits, w.kivi_R)
    kvc.kvc_append_quant(cache, K[:, :, :w.T - 1].contiguous(), V[:, :, :w.T - 1].contiguous())
    kvc.kvc_append_quant(cache, K[:, :, w.T - 1:].contiguous(), V[:, :, w.T - 1:].contiguous())
    o, lse = _attend(kvc, cache, q)
    rng = np.random.default_rng(1)
    gq = w.Hq // w.Hkv
    for b in sorted(set(rng.integers(0, w.B, 4).tolist()) | {w.B - 1}):
        hk = int(rng.integers(0, w.Hkv))
        Kb, Vb = np16(K[b, hk]), np16(V[b, hk])
        n_q = orc.kivi_nq(w.T, w.kivi_R)
        qz = orc.kivi_quantize_unit(Kb[:n_q], Vb[:n_q], n_q, bits)
        kb, vb = orc.kivi_pack_unit(qz, w.D, bits)
        assert np.array_equal(cache.k_blocks[b, hk].cpu().numpy(), kb)
        assert np.array_equal(cache.v_blocks[b, hk].cpu().numpy(), vb)
        ref, _ = orc.kivi_attend_unit(np16(q[b, hk * gq:(hk + 1) * gq]), Kb, Vb, w.T, w.kivi_R,
                                      bits, qz=qz)
        assert_o_close(np16(o[b, hk * gq:(hk + 1) * gq]), ref, what=f"b={b} hk={hk}")
    assert device_status_clean(kvc)


def test_capacity_overflow_is_flagged(kvc):
    cache = kvc.QuantCache.empty(1, 1, 32, 64, 4, 16)
    k = torch.zeros(1, 1, 100, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(kvc.KvcError) as e:       # more new tokens than the cache can hold
        kvc.kvc_append_quant(cache, k, k)
    assert e.value.status == kvc.KVC_ERR_CAPACITY
    k = torch.zeros(1, 1, 40, 64, dtype=torch.float16, device="cuda")
    kvc.kvc_append_quant(cache, k, k)            # T = 40: everything in the residual
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status() == 0
    kvc.kvc_append_quant(cache, k, k)            # T = 80: n_q = 64 > Cq = 32, seen on the device
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status() & kvc.KVC_DEV_CAPACITY
    assert kvc.kvc_read_device_status() == 0     # reading clears it


@pytest.mark.parametrize("bits", [4, 2])
def test_long_single_sequence_auto_splits(kvc, orc, bits):
    """One sequence of the heavy-load head layout (GQA 64/8, D 128) at 16384 tokens, in the
    launch configuration of the throughput profile grid (automatic splits): every unit's blocks
    are bit-exact and its attention matches the oracle."""
    B, Hq, Hkv, D, T, R = 1, 64, 8, 128, 16384, 128
    g = torch.Generator().manual_seed(T + bits)
    K = torch.randn(B, Hkv, T, D, generator=g).half()
    V = torch.randn(B, Hkv, T, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    n_q = orc.kivi_nq(T, R)
    cache = kvc.QuantCache.empty(B, Hkv, n_q, D, bits, R)
    kvc.kvc_append_quant(cache, K.cuda(), V.cuda())
    o, _ = _attend(kvc, cache, q.cuda())
    gq = Hq // Hkv
    for hk in range(Hkv):
        Kb, Vb = np16(K[0, hk]), np16(V[0, hk])
        qz = orc.kivi_quantize_unit(Kb[:n_q], Vb[:n_q], n_q, bits)
        kb, vb = orc.kivi_pack_unit(qz, D, bits)
        assert np.array_equal(cache.k_blocks[0, hk].cpu().numpy(), kb)
        assert np.array_equal(cache.v_blocks[0, hk].cpu().numpy(), vb)
        ref, _ = orc.kivi_attend_unit(np16(q[0, hk * gq:(hk + 1) * gq]), Kb, Vb, T, R, bits, qz=qz)
        assert_o_close(np16(o[0, hk * gq:(hk + 1) * gq]), ref, what=f"hk={hk}")
    assert device_status_clean(kvc)


def _crafted_kv(rng, T, D, kind):
    """[T, D] fp16 tensors whose 32-token K groups and 32-channel V groups hit the quantiser's
    edge cases: 'wide' spans 10^-6 .. 10^4 per 32x32 block (subnormal scales, large ranges),
    'coarse' multiples of 0.25 (exact ties at half-steps), 'flat' constant and signed-zero
    groups mixed with ordinary ones (degenerate scale 0, zero point -0)."""
    if kind == "wide":
        x = rng.standard_normal((T, D)) * np.repeat(np.repeat(
            10.0 ** rng.uniform(-6, 4, (T // 32, D // 32)), 32, 0), 32, 1)
    elif kind == "coarse":
        x = rng.integers(-8, 8, (T, D)) * 0.25
    else:
        x = rng.standard_normal((T, D))
        x[:32] = 1.5                                   # constant K and V groups
        x[32:64, :32] = -0.0
        x[32:64, 32:64] = np.where(rng.random((32, 32)) < 0.5, -0.0, 0.0)
        x[64:96, :] = np.where(rng.random((32, D)) < 0.1, rng.standard_normal((32, D)), 0.0)
    return x.astype(np.float16)


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("kind", ["wide", "coarse", "flat"])
def test_pack_bit_exact_crafted(kvc, orc, bits, kind):
    """Bulk pack of crafted groups (wide-range, tie-heavy, degenerate) is bit-exact."""
    rng = np.random.default_rng(bits * 7 + len(kind))
    B, Hkv, D, T, R = 2, 2, 128, 288, 32
    K = np.stack([np.stack([_crafted_kv(rng, T, D, kind) for _ in range(Hkv)]) for _ in range(B)])
    V = np.stack([np.stack([_crafted_kv(rng, T, D, kind) for _ in range(Hkv)]) for _ in range(B)])
    n_q = orc.kivi_nq(T, R)
    cache = kvc.QuantCache.empty(B, Hkv, n_q, D, bits, R)
    kvc.kvc_append_quant(cache, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    torch.cuda.synchronize()
    for b in range(B):
        for hk in range(Hkv):
            qz = orc.kivi_quantize_unit(K[b, hk, :n_q], V[b, hk, :n_q], n_q, bits)
            kb, vb = orc.kivi_pack_unit(qz, D, bits)
            assert np.array_equal(cache.k_blocks[b, hk].cpu().numpy(), kb), (b, hk)
            assert np.array_equal(cache.v_blocks[b, hk].cpu().numpy(), vb), (b, hk)
    assert device_status_clean(kvc)


def _ragged_quant_cache(kvc, K, V, lens, bits, R, Cq, gear=False):
    """A KIVI (or GEAR) cache whose sequence b holds the first lens[b] tokens of K/V
    [B, Hkv, T, D] (host), each appended through a one-sequence view of the batch."""
    B = K.shape[0]
    cache = kvc.QuantCache.empty(B, K.shape[1], Cq, K.shape[3], bits, R, gear=gear)
    for b in range(B):
        if lens[b] == 0:
            continue
        view = kvc.QuantCache(k_blocks=cache.k_blocks[b:b + 1], v_blocks=cache.v_blocks[b:b + 1],
                              k_res=cache.k_res[b:b + 1], v_res=cache.v_res[b:b + 1],
                              len=cache.len[b:b + 1], bits=bits, R=R,
                              k_gear=cache.k_gear[b:b + 1] if gear else None,
                              v_gear=cache.v_gear[b:b + 1] if gear else None)
        kvc.kvc_append_quant(view, K[b:b + 1, :, :lens[b]].cuda().contiguous(),
                             V[b:b + 1, :, :lens[b]].cuda().contiguous())
    torch.cuda.synchronize()
    assert cache.len.cpu().tolist() == list(lens)
    return cache


def _check_ragged(orc, q, K, V, lens, R, bits, o, lse):
    gq = q.shape[1] // K.shape[1]
    for b, T in enumerate(lens):
        for hk in range(K.shape[1]):
            og = np16(o[b, hk * gq:(hk + 1) * gq])
            lg = lse[b, hk * gq:(hk + 1) * gq].cpu().numpy()
            if T == 0:   # an empty softmax: no mass
                assert not og.astype(np.float64).any() and np.isneginf(lg).all()
                continue
            ref, ref_lse = orc.kivi_attend_unit(np16(q[b, hk * gq:(hk + 1) * gq]),
                                                np16(K[b, hk]), np16(V[b, hk]), T, R, bits)
            assert_o_close(og, ref, what=f"T={T} hk={hk}")
            np.testing.assert_allclose(lg, ref_lse, atol=KIVI_LSE_TOL, rtol=0)


@pytest.mark.parametrize("bits,splits", [(4, 0), (2, 0), (4, 3)])
def test_ragged_edge_lengths(kvc, orc, bits, splits):
    """One batch whose sequences sit at the edges of the flush rule: empty, a single token,
    R - 1, R (ring full, nothing quantised), R + 31 (one short of a flush), R + 32 (first
    group), R + 33 and R + 100."""
    D, Hq, Hkv, R = 128, 8, 2, 64
    lens = [0, 1, R - 1, R, R + 31, R + 32, R + 33, R + 100]
    g = torch.Generator().manual_seed(bits + 10 * splits)
    T = max(lens)
    K = (torch.randn(len(lens), Hkv, T, D, generator=g) * 2).half()
    V = torch.randn(len(lens), Hkv, T, D, generator=g).half()
    q = torch.randn(len(lens), Hq, D, generator=g).half()
    cache = _ragged_quant_cache(kvc, K, V, lens, bits, R, 128)
    o, lse = _attend(kvc, cache, q.cuda(), splits)
    _check_ragged(orc, q, K, V, lens, R, bits, o, lse)
    assert device_status_clean(kvc)


@pytest.mark.parametrize("bits", [2, 4])
def test_tail_units_split_over_idle_ctas(kvc, orc, bits):
    """The automatic plan when the persistent CTAs (three per SM) take whole units in rounds and
    the last round fills few of them: 3 x SMs + 10 units, so the last 10 units are split four
    ways (partials merged afterwards) and the rest run whole.  Ragged lengths; every unit is
    compared with the single-split launch, the split units and some whole ones with the
    oracle."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    D, Hq, Hkv, R, Cq = 128, 4, 2, 32, 512
    units = 3 * n_sm + 10
    B = units // Hkv
    pattern = [575, 1, 400, 544, 100, 0, 33, 64]
    lens = [pattern[b % len(pattern)] for b in range(B)]
    g = torch.Generator().manual_seed(40 + bits)
    T = max(lens)
    K = torch.randn(B, Hkv, T, D, generator=g).half()
    V = torch.randn(B, Hkv, T, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half()
    cache = _ragged_quant_cache(kvc, K, V, lens, bits, R, Cq)
    qd = q.cuda()
    assert kvc.kvc_workspace_size(cache, qd) > 0            # the tail plan is in use
    o, lse = _attend(kvc, cache, qd)
    o1, lse1 = _attend(kvc, cache, qd, 1)
    assert_o_close(np16(o), np16(o1).astype(np.float64), what="auto vs one split")
    fin = torch.isfinite(lse1)
    assert torch.equal(fin, torch.isfinite(lse))
    assert torch.allclose(lse[fin], lse1[fin], atol=KIVI_LSE_TOL, rtol=0)
    gq = Hq // Hkv
    first_split = units - units % (3 * n_sm)
    check = sorted({u // Hkv for u in range(first_split, units)} | {0, 1, first_split // Hkv - 1})
    for b in check:
        for hk in range(Hkv):
            if lens[b] == 0:
                assert not np16(o[b, hk * gq:(hk + 1) * gq]).astype(np.float64).any()
                continue
            ref, ref_lse = orc.kivi_attend_unit(np16(q[b, hk * gq:(hk + 1) * gq]), np16(K[b, hk]),
                                                np16(V[b, hk]), lens[b], R, bits)
            assert_o_close(np16(o[b, hk * gq:(hk + 1) * gq]), ref, what=f"b={b} hk={hk}")
            np.testing.assert_allclose(lse[b, hk * gq:(hk + 1) * gq].cpu().numpy(), ref_lse,
                                       atol=KIVI_LSE_TOL, rtol=0)
    assert device_status_clean(kvc)


def test_tail_units_split_over_idle_ctas_gear(kvc):
    """The same plan for a GEAR cache, whose kernel keeps two CTAs per SM: 2 x SMs + 6 units;
    every unit matches the single-split launch (itself checked against the GEAR oracle in
    tests/test_gpu_gear.py)."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    D, Hq, Hkv, R, Cq = 128, 8, 2, 32, 256
    units = 2 * n_sm + 6
    B = units // Hkv
    pattern = [287, 1, 200, 256, 64, 0, 40]
    lens = [pattern[b % len(pattern)] for b in range(B)]
    g = torch.Generator().manual_seed(77)
    T = max(lens)
    K = torch.randn(B, Hkv, T, D, generator=g).half()
    V = torch.randn(B, Hkv, T, D, generator=g).half()
    q = torch.randn(B, Hq, D, generator=g).half().cuda()
    cache = _ragged_quant_cache(kvc, K, V, lens, 4, R, Cq, gear=True)
    assert kvc.kvc_workspace_size(cache, q) > 0            # the tail plan is in use
    o, lse = _attend(kvc, cache, q)
    o1, lse1 = _attend(kvc, cache, q, 1)
    assert_o_close(np16(o), np16(o1).astype(np.float64), what="auto vs one split")
    fin = torch.isfinite(lse1)
    assert torch.equal(fin, torch.isfinite(lse))
    assert torch.allclose(lse[fin], lse1[fin], atol=KIVI_LSE_TOL, rtol=0)
    assert device_status_clean(kvc)
