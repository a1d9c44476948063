"""CPU-only checks of the C ABI: the library loads, exports every function that
include/kvc.h declares, and answers host-side queries (no kernel is launched)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvc():
    from kv_cache_compression_split_gb300 import build
    build.build()
    import kv_cache_compression_split_gb300 as k
    k.lib()
    return k


def _declared():
    hdr = open(os.path.join(ROOT, "include", "kvc.h")).read()
    return sorted(set(re.findall(r"KVC_API\s+[\w\s\*]+?\b(kvc_\w+)\s*\(", hdr)))


def test_every_declared_symbol_is_exported(kvc):
    names = _declared()
    assert len(names) >= 12
    lib = ctypes.CDLL(kvc.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name


def test_host_queries(kvc):
    assert kvc.kvc_kivi_block_bytes(128, 4) == 32 * 128 * 4 // 8 + 4 * 128 == 2560
    assert kvc.kvc_kivi_block_bytes(128, 2) == 1536
    assert kvc.kvc_kivi_block_bytes(64, 4) == 1280
    assert kvc.kvc_kivi_block_bytes(96, 4) == 0      # unsupported head dim
    assert kvc.kvc_kivi_block_bytes(128, 3) == 0     # unsupported width
    assert "INVALID_ARG" in kvc.kvc_status_string(kvc.KVC_ERR_INVALID_ARG)
    assert kvc.kvc_status_string(kvc.KVC_OK) == "KVC_OK"


def test_null_arguments_are_rejected_without_touching_a_gpu(kvc):
    lib = kvc.lib()
    assert lib.kvc_append(None, None, None, 1, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_append_quant(None, None, None, 1, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_decode_attend(None, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_h2o_accumulate(None, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_h2o_evict(None, None, 1, 1, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_stream_evict(None, 1, 1, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_stream_append(None, None, None, 1, 1, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_h2o_decode_step(None, None, 8, None, None, None, None, None, 64, 448, 0.0,
                                   None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_stream_decode_step(None, 8, None, None, None, None, None, 64, 448,
                                      None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_random_evict(None, 0, 0.5, 1, 0, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_read_device_status(None, None) == kvc.KVC_ERR_INVALID_ARG
    # a descriptor with an unsupported head dim (pointers are never dereferenced on the host)
    d = kvc.SlotCacheDesc(1, 1, 96, 16, 16, 16, 16, 16, 16)
    assert lib.kvc_stream_evict(ctypes.byref(d), 1, 1, None) == kvc.KVC_ERR_UNSUPPORTED
    d = kvc.SlotCacheDesc(1, 1, 128, 16, 16, 17, 16, 16, 16)     # misaligned V
    assert lib.kvc_stream_evict(ctypes.byref(d), 1, 1, None) == kvc.KVC_ERR_INVALID_ARG
    q = kvc.QuantCacheDesc(1, 1, 128, 3, 16, 32, 16, 16, 16, 16, 16)
    assert lib.kvc_append_quant(ctypes.byref(q), None, None, 0, None) == kvc.KVC_ERR_UNSUPPORTED
    # paged layout: C must be whole pages and the pool must not be empty
    d = kvc.SlotCacheDesc(1, 1, 128, 100, 16, 16, 16, 16, 16, 16, 4)
    assert lib.kvc_stream_evict(ctypes.byref(d), 1, 1, None) == kvc.KVC_ERR_INVALID_ARG
    d = kvc.SlotCacheDesc(1, 1, 128, 128, 16, 16, 16, 16, 16, 16, 0)
    assert lib.kvc_stream_evict(ctypes.byref(d), 1, 1, None) == kvc.KVC_ERR_INVALID_ARG
    # batched H2O eviction: null cache, and a trigger that is not positive
    assert lib.kvc_h2o_evict_when(None, None, 64, 448, 563, None) == kvc.KVC_ERR_INVALID_ARG
    d = kvc.SlotCacheDesc(1, 1, 128, 16, 16, 16, 16, 16, 16)
    assert lib.kvc_h2o_evict_when(ctypes.byref(d), 16, 64, 448, 0, None) == kvc.KVC_ERR_INVALID_ARG
    # decay outside {0} U (0, 1) is refused before anything is launched
    for bad in (1.0, 1.5, -0.1, float("nan")):
        h = kvc._h2o_args(kvc.KVC_H2O_DECODE, 1, 1, 1, 128, 16, None, decay=bad)
        h.scores = h.logits = h.lse = h.n = 16
        assert lib.kvc_h2o_accumulate(ctypes.byref(h), None) == kvc.KVC_ERR_INVALID_ARG, bad
        a = kvc.AttendArgs()
        a.kind, a.Hq, a.q, a.o, a.slots = kvc.KVC_KIND_SLOTS, 1, 16, 16, ctypes.pointer(d)
        a.logits = a.lse = a.h2o_scores = 16
        a.h2o_decay = bad
        assert lib.kvc_decode_attend(ctypes.byref(a), None) == kvc.KVC_ERR_INVALID_ARG, bad
    # q and o are 16-byte aligned like every other pointer (the split combine writes o
    # 8 bytes at a time)
    a = kvc.AttendArgs()
    a.kind, a.Hq, a.q, a.o, a.slots = kvc.KVC_KIND_SLOTS, 1, 16, 18, ctypes.pointer(d)
    assert lib.kvc_decode_attend(ctypes.byref(a), None) == kvc.KVC_ERR_INVALID_ARG
    a.q, a.o = 24, 16
    assert lib.kvc_decode_attend(ctypes.byref(a), None) == kvc.KVC_ERR_INVALID_ARG
    # fused H2O with the logits on chip: at most one cluster of 8 splits, each split within
    # the on-chip bound of KVC_H2O_ONCHIP_MAX_SLOTS slots
    a = kvc.AttendArgs()
    a.kind, a.Hq, a.q, a.o, a.slots = kvc.KVC_KIND_SLOTS, 1, 16, 16, ctypes.pointer(d)
    a.lse = a.h2o_scores = 16
    a.num_splits = 9
    assert lib.kvc_decode_attend(ctypes.byref(a), None) == kvc.KVC_ERR_INVALID_ARG
    a.num_splits = 1
    big = kvc.SlotCacheDesc(1, 1, 128, kvc.H2O_ONCHIP_MAX_SLOTS + 64, 16, 16, 16, 16, 16)
    a.slots = ctypes.pointer(big)
    assert lib.kvc_decode_attend(ctypes.byref(a), None) == kvc.KVC_ERR_UNSUPPORTED
    a.num_splits = 2                 # two splits of at most 1024 slots: planned, no workspace
    assert lib.kvc_workspace_size(ctypes.byref(a)) == 0
    huge = kvc.SlotCacheDesc(1, 1, 128, 8 * kvc.H2O_ONCHIP_MAX_SLOTS + 64, 16, 16, 16, 16, 16)
    a.slots = ctypes.pointer(huge)
    a.num_splits = 0                 # would need 9 splits
    assert lib.kvc_decode_attend(ctypes.byref(a), None) == kvc.KVC_ERR_UNSUPPORTED
    a.logits = 16                    # with a logits array any capacity and split count is fine
    a.num_splits = 12                # more splits than a cluster: partials in a workspace
    assert lib.kvc_workspace_size(ctypes.byref(a)) > 0


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "kv_cache_compression_split_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f), errors="ignore").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "oracle.c" not in src and "liboracle" not in src, f


def test_binding_rejects_host_and_strided_tensors():
    """The binding hands only contiguous tensors of the current CUDA device to the library: a
    host tensor's address would otherwise reach a kernel as if it were device memory."""
    import torch
    import kv_cache_compression_split_gb300 as kvc
    cache = kvc.SlotCache.empty(1, 1, 64, 64, device="cpu")
    q = torch.zeros(1, 1, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        kvc.kvc_decode_attend(cache, q, torch.empty_like(q))
    with pytest.raises(ValueError, match="CUDA tensors"):
        kvc.kvc_append(cache, torch.zeros(1, 1, 1, 64, dtype=torch.float16),
                       torch.zeros(1, 1, 1, 64, dtype=torch.float16))


def test_prefill_args_carry_the_row_normalisers(kvc):
    """The prefill arguments pass the optional row normalisers through to the C struct (NULL
    when absent), and a prefill without workspace is refused before anything is launched."""
    h = kvc._h2o_args(kvc.KVC_H2O_PREFILL, 1, 8, 1, 128, 300, 16, lse=4096, L=300, qp=16, kp=16,
                      kp_cap=300)
    assert h.lse == 4096 and h.mode == kvc.KVC_H2O_PREFILL
    h2 = kvc._h2o_args(kvc.KVC_H2O_PREFILL, 1, 8, 1, 128, 300, 16, L=300, qp=16, kp=16,
                       kp_cap=300)
    assert h2.lse is None
    lib = kvc.lib()
    assert lib.kvc_h2o_accumulate(ctypes.byref(h), None) == kvc.KVC_ERR_WORKSPACE


def test_cache_objects_pickle_and_copy_without_their_descriptor():
    """A cache object keeps its ctypes descriptor between calls; pickling or copying it
    leaves that out (ctypes pointers do not pickle), and the copy rebuilds its own."""
    import copy
    import pickle
    import kv_cache_compression_split_gb300 as kvc
    cache = kvc.SlotCache.empty(1, 2, 64, 64, device="cpu")
    d = kvc.SlotCacheDesc()
    cache.__dict__.update(_desc=d, _desc_key=("k",), _desc_p=ctypes.pointer(d))
    back = pickle.loads(pickle.dumps(cache))
    assert "_desc" not in back.__dict__ and back.K.shape == cache.K.shape
    dup = copy.copy(cache)
    assert "_desc_p" not in dup.__dict__ and dup.K is cache.K
    q = kvc.QuantCache.empty(1, 2, 256, 64, 4, 128, device="cpu")
    q.__dict__.update(_desc=kvc.QuantCacheDesc(), _desc_key=("k",))
    assert "_desc" not in pickle.loads(pickle.dumps(q)).__dict__
