"""Python binding of libkvc.so -- the GB300 compressed-KV decode library.

This module only marshals arguments: it builds the C descriptor structs from
torch tensors (device memory owned by the caller) and calls the C ABI declared
in include/kvc.h with the same function names.  Every step of the path runs in
the library's CUDA kernels; there is no Python or CPU fallback -- if the
library is missing, importing a function raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvc.so")
_lib = None
_lock = threading.Lock()

KVC_OK, KVC_ERR_INVALID_ARG, KVC_ERR_UNSUPPORTED, KVC_ERR_CAPACITY = 0, 1, 2, 3
KVC_ERR_WORKSPACE, KVC_ERR_CUDA, KVC_ERR_DEVICE = 4, 5, 6
KVC_DEV_CAPACITY, KVC_DEV_TIMEOUT = 0x1, 0x2
KVC_KIND_SLOTS, KVC_KIND_KIVI = 0, 1
KVC_H2O_DECODE, KVC_H2O_PREFILL = 0, 1
KIVI_GROUP = 32
PAGE_SLOTS = 64            # KVC_PAGE_SLOTS: slots per page of the paged layout
KIVI_PAGE_GROUPS = 4       # KVC_KIVI_PAGE_GROUPS: 32-token groups per KIVI page
H2O_ONCHIP_MAX_SLOTS = 1024   # KVC_H2O_ONCHIP_MAX_SLOTS: fused H2O with logits kept on chip
KVC_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class KvcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kvc_status_string(status)}")


class SlotCacheDesc(C.Structure):
    _fields_ = [("B", C.c_int), ("Hkv", C.c_int), ("D", C.c_int), ("C", C.c_int),
                ("K", C.c_void_p), ("V", C.c_void_p), ("pos", C.c_void_p), ("n", C.c_void_p),
                ("seqlen", C.c_void_p), ("block_table", C.c_void_p), ("num_pages", C.c_int)]


class QuantCacheDesc(C.Structure):
    _fields_ = [("B", C.c_int), ("Hkv", C.c_int), ("D", C.c_int), ("bits", C.c_int),
                ("R", C.c_int), ("Cq", C.c_int), ("k_blocks", C.c_void_p),
                ("v_blocks", C.c_void_p), ("k_res", C.c_void_p), ("v_res", C.c_void_p),
                ("len", C.c_void_p), ("block_table", C.c_void_p), ("num_pages", C.c_int),
                ("k_gear", C.c_void_p), ("v_gear", C.c_void_p)]


class AttendArgs(C.Structure):
    _fields_ = [("kind", C.c_int), ("Hq", C.c_int), ("q", C.c_void_p), ("o", C.c_void_p),
                ("slots", C.POINTER(SlotCacheDesc)), ("quant", C.POINTER(QuantCacheDesc)),
                ("logits", C.c_void_p), ("lse", C.c_void_p), ("workspace", C.c_void_p),
                ("workspace_bytes", C.c_size_t), ("num_splits", C.c_int),
                ("softmax_scale", C.c_float), ("h2o_scores", C.c_void_p),
                ("h2o_decay", C.c_float)]


class H2OArgs(C.Structure):
    _fields_ = [("mode", C.c_int), ("B", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int),
                ("D", C.c_int), ("C", C.c_int), ("scores", C.c_void_p), ("logits", C.c_void_p),
                ("lse", C.c_void_p), ("n", C.c_void_p), ("L", C.c_int), ("qp", C.c_void_p),
                ("kp", C.c_void_p), ("kp_cap", C.c_int), ("workspace", C.c_void_p),
                ("workspace_bytes", C.c_size_t), ("softmax_scale", C.c_float),
                ("decay", C.c_float)]


def lib():
    """Load libkvc.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with "
                                  "`python -m kv_cache_compression_split_gb300.build`")
            L = C.CDLL(LIB_PATH)
            P, i, st = C.c_void_p, C.c_int, C.c_int
            sig = {
                "kvc_kivi_block_bytes": (C.c_size_t, [i, i]),
                "kvc_gear_side_bytes": (C.c_size_t, [i]),
                "kvc_append": (st, [C.POINTER(SlotCacheDesc), P, P, i, P]),
                "kvc_append_quant": (st, [C.POINTER(QuantCacheDesc), P, P, i, P]),
                "kvc_workspace_size": (C.c_size_t, [C.POINTER(AttendArgs)]),
                "kvc_decode_attend": (st, [C.POINTER(AttendArgs), P]),
                "kvc_decode_attend_noalloc": (st, [C.POINTER(AttendArgs), P]),
                "kvc_h2o_workspace_size": (C.c_size_t, [C.POINTER(H2OArgs)]),
                "kvc_h2o_accumulate": (st, [C.POINTER(H2OArgs), P]),
                "kvc_h2o_evict": (st, [C.POINTER(SlotCacheDesc), P, i, i, P]),
                "kvc_h2o_evict_when": (st, [C.POINTER(SlotCacheDesc), P, i, i, i, P]),
                "kvc_stream_evict": (st, [C.POINTER(SlotCacheDesc), i, i, P]),
                "kvc_stream_append": (st, [C.POINTER(SlotCacheDesc), P, P, i, i, P]),
                "kvc_h2o_decode_step": (st, [C.POINTER(SlotCacheDesc), P, i, P, P, P, P, P, i, i,
                                             C.c_float, P]),
                "kvc_stream_decode_step": (st, [C.POINTER(SlotCacheDesc), i, P, P, P, P, P, i, i,
                                                P]),
                "kvc_random_evict": (st, [C.POINTER(SlotCacheDesc), i, C.c_double, C.c_uint64,
                                          C.c_uint32, P]),
                "kvc_status_string": (C.c_char_p, [i]),
                "kvc_read_device_status": (st, [C.POINTER(C.c_int), P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


# ----------------------------------------------------------------------------- helpers

def _ptr(t):
    """Device address of tensor t for a descriptor field.  Every tensor handed to the library
    must be contiguous and live on the current CUDA device: a host tensor's address given to
    a kernel would be read as device memory (or, where the GPU can reach host memory, read
    silently)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"kvc: tensor on {t.device}; the library takes CUDA tensors")
    if t.get_device() != torch.cuda.current_device() or not t.is_contiguous():
        if t.device.index != torch.cuda.current_device():
            raise ValueError(f"kvc: tensor on {t.device}, expected the current device "
                             f"cuda:{torch.cuda.current_device()}")
        raise ValueError("kvc: tensor arguments must be contiguous")
    return t.data_ptr()


# torch's raw current-stream query, where this torch version has it (a few hundred ns
# against a few microseconds for torch.cuda.current_stream())
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _desc_key(tensors):
    """What a cache descriptor depends on: each field tensor's address, device, shape and
    strides (None for an absent field)."""
    return tuple(None if t is None else (t.data_ptr(), t.get_device(), t.shape, t.stride())
                 for t in tensors)


_DESC_CACHE_KEYS = ("_desc", "_desc_key", "_desc_p")


def _state_without_desc(obj):
    """A cache object's state for pickling and copying: its fields, without the kept ctypes
    descriptor (rebuilt on the next call; ctypes pointers do not pickle)."""
    state = dict(obj.__dict__)
    for k in _DESC_CACHE_KEYS:
        state.pop(k, None)
    return state



def _stream(stream):
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != KVC_OK:
        raise KvcError(status, where)


# ----------------------------------------------------------------------------- C ABI, same names

def kvc_status_string(status: int) -> str:
    return lib().kvc_status_string(int(status)).decode()


def kvc_kivi_block_bytes(D: int, bits: int) -> int:
    return int(lib().kvc_kivi_block_bytes(D, bits))


def kvc_append(cache: "SlotCache", k_new, v_new, stream=None):
    d = cache.desc()
    _check(lib().kvc_append(C.byref(d), _ptr(k_new), _ptr(v_new), int(k_new.shape[2]),
                            _stream(stream)), "kvc_append")


def kvc_append_quant(cache: "QuantCache", k_new, v_new, stream=None):
    d = cache.desc()
    _check(lib().kvc_append_quant(C.byref(d), _ptr(k_new), _ptr(v_new), int(k_new.shape[2]),
                                  _stream(stream)), "kvc_append_quant")


def _attend_args(cache, q, o, logits=None, lse=None, workspace=None, num_splits=0, scale=0.0,
                 h2o_scores=None, h2o_decay=0.0, shape_only=False):
    a = AttendArgs()
    keep = []
    d = cache.desc()
    keep.append(d)
    if isinstance(cache, SlotCache):
        a.kind = KVC_KIND_SLOTS
        a.slots = cache.__dict__["_desc_p"]
    else:
        a.kind = KVC_KIND_KIVI
        a.quant = cache.__dict__["_desc_p"]
    a.Hq = int(q.shape[1])
    # a size query reads only q's shape (the library plans from the dimensions)
    a.q, a.o = (None, None) if shape_only else (_ptr(q), _ptr(o))
    a.logits, a.lse = _ptr(logits), _ptr(lse)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.num_splits = int(num_splits)
    a.softmax_scale = float(scale)
    a.h2o_scores = _ptr(h2o_scores)
    a.h2o_decay = float(h2o_decay)
    return a, keep


def kvc_gear_side_bytes(D: int) -> int:
    return int(lib().kvc_gear_side_bytes(D))


def kvc_workspace_size(cache, q, num_splits: int = 0) -> int:
    a, _keep = _attend_args(cache, q, None, num_splits=num_splits, shape_only=True)
    return int(lib().kvc_workspace_size(C.byref(a)))


def kvc_decode_attend(cache, q, o, logits=None, lse=None, workspace=None, num_splits: int = 0,
                      softmax_scale: float = 0.0, h2o_scores=None, h2o_decay: float = 0.0,
                      stream=None):
    a, _keep = _attend_args(cache, q, o, logits, lse, workspace, num_splits, softmax_scale,
                            h2o_scores, h2o_decay)
    _check(lib().kvc_decode_attend(C.byref(a), _stream(stream)), "kvc_decode_attend")


def kvc_decode_attend_noalloc(cache, q, o, logits=None, lse=None, num_splits: int = 0,
                              softmax_scale: float = 0.0, h2o_scores=None, h2o_decay: float = 0.0,
                              stream=None):
    """kvc_decode_attend without a caller workspace: for callers that cannot allocate device
    memory on their decode path, the split scratch comes from a fixed array the library owns
    (KVC_NOALLOC_SCRATCH_BYTES per GPU).  Calls that may overlap on the GPU race on it."""
    a, _keep = _attend_args(cache, q, o, logits, lse, None, num_splits, softmax_scale,
                            h2o_scores, h2o_decay)
    _check(lib().kvc_decode_attend_noalloc(C.byref(a), _stream(stream)),
           "kvc_decode_attend_noalloc")


def _h2o_args(mode, B, Hq, Hkv, D, Cc, scores, logits=None, lse=None, n=None, L=0, qp=None,
              kp=None, kp_cap=0, workspace=None, scale=0.0, decay=0.0):
    a = H2OArgs()
    a.mode, a.B, a.Hq, a.Hkv, a.D, a.C = mode, B, Hq, Hkv, D, Cc
    a.scores, a.logits, a.lse, a.n = _ptr(scores), _ptr(logits), _ptr(lse), _ptr(n)
    a.L, a.qp, a.kp, a.kp_cap = int(L), _ptr(qp), _ptr(kp), int(kp_cap)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.softmax_scale = float(scale)
    a.decay = float(decay)
    return a


def kvc_h2o_workspace_size(B: int, Hq: int, L: int) -> int:
    a = _h2o_args(KVC_H2O_PREFILL, B, Hq, 1, 128, 1, None, L=L)
    return int(lib().kvc_h2o_workspace_size(C.byref(a)))


def kvc_h2o_accumulate_decode(cache: "SlotCache", scores, logits, lse, Hq: int,
                              decay: float = 0.0, stream=None):
    a = _h2o_args(KVC_H2O_DECODE, cache.B, Hq, cache.Hkv, cache.D, cache.C, scores, logits, lse,
                  cache.n, decay=decay)
    _check(lib().kvc_h2o_accumulate(C.byref(a), _stream(stream)), "kvc_h2o_accumulate")


def kvc_h2o_accumulate_prefill(qp, kp, scores, workspace, L: int, lse=None, stream=None):
    """lse: optional [B, Hq, L] fp32 natural-log row normalisers (skips the row pass)."""
    B, Hq, _, D = qp.shape
    _, Hkv, kp_cap, _ = kp.shape
    a = _h2o_args(KVC_H2O_PREFILL, B, Hq, Hkv, D, int(scores.shape[-1]), scores, lse=lse, L=L,
                  qp=qp, kp=kp, kp_cap=kp_cap, workspace=workspace)
    _check(lib().kvc_h2o_accumulate(C.byref(a), _stream(stream)), "kvc_h2o_accumulate")


def kvc_h2o_accumulate(args: H2OArgs, stream=None):
    _check(lib().kvc_h2o_accumulate(C.byref(args), _stream(stream)), "kvc_h2o_accumulate")


def kvc_h2o_evict(cache: "SlotCache", scores, n_heavy: int, n_recent: int, stream=None):
    d = cache.desc()
    _check(lib().kvc_h2o_evict(C.byref(d), _ptr(scores), n_heavy, n_recent, _stream(stream)),
           "kvc_h2o_evict")


def kvc_h2o_evict_when(cache: "SlotCache", scores, n_heavy: int, n_recent: int, trigger: int,
                       stream=None):
    d = cache.desc()
    _check(lib().kvc_h2o_evict_when(C.byref(d), _ptr(scores), n_heavy, n_recent, int(trigger),
                                    _stream(stream)), "kvc_h2o_evict_when")


def kvc_stream_evict(cache: "SlotCache", n_sink: int, n_recent: int, stream=None):
    d = cache.desc()
    _check(lib().kvc_stream_evict(C.byref(d), n_sink, n_recent, _stream(stream)),
           "kvc_stream_evict")


def kvc_stream_append(cache: "SlotCache", k_new, v_new, n_sink: int, n_recent: int, stream=None):
    """One StreamingLLM decode token per sequence ([B, Hkv, 1, D]); the token leaving the
    window gives up its slot (see kvc.h)."""
    if int(k_new.shape[2]) != 1 or int(v_new.shape[2]) != 1:
        raise ValueError("kvc_stream_append takes one token per sequence")
    d = cache.desc()
    _check(lib().kvc_stream_append(C.byref(d), _ptr(k_new), _ptr(v_new), n_sink, n_recent,
                                   _stream(stream)), "kvc_stream_append")


def kvc_h2o_decode_step(cache: "SlotCache", scores, q, k_new, v_new, o, lse=None,
                        n_heavy: int = 64, n_recent: int = 448, decay: float = 0.0, stream=None):
    """One H2O decode step (append + attention + score update + eviction) in one launch."""
    d = cache.desc()
    _check(lib().kvc_h2o_decode_step(C.byref(d), _ptr(scores), int(q.shape[1]), _ptr(q),
                                     _ptr(k_new), _ptr(v_new), _ptr(o), _ptr(lse), n_heavy,
                                     n_recent, float(decay), _stream(stream)),
           "kvc_h2o_decode_step")


def kvc_stream_decode_step(cache: "SlotCache", q, k_new, v_new, o, lse=None, n_sink: int = 64,
                           n_recent: int = 448, stream=None):
    """One StreamingLLM decode step (append into the leaving token's slot + attention) in one
    launch."""
    d = cache.desc()
    _check(lib().kvc_stream_decode_step(C.byref(d), int(q.shape[1]), _ptr(q), _ptr(k_new),
                                        _ptr(v_new), _ptr(o), _ptr(lse), n_sink, n_recent,
                                        _stream(stream)), "kvc_stream_decode_step")


def kvc_random_evict(cache: "SlotCache", prompt_len: int, keep_ratio: float, seed: int,
                     epoch: int, stream=None):
    d = cache.desc()
    _check(lib().kvc_random_evict(C.byref(d), prompt_len, float(keep_ratio),
                                  seed & (2**64 - 1), epoch & 0xffffffff, _stream(stream)),
           "kvc_random_evict")


def kvc_read_device_status(stream=None) -> int:
    out = C.c_int(0)
    st = lib().kvc_read_device_status(C.byref(out), _stream(stream))
    if st not in (KVC_OK, KVC_ERR_DEVICE):
        raise KvcError(st, "kvc_read_device_status")
    return out.value


# ----------------------------------------------------------------------------- cache holders

@dataclass
class SlotCache:
    """fp16 slot cache in device memory (layout documented in include/kvc.h).  Dense layout:
    K, V [B, Hkv, C, D].  Paged layout: K, V are page pools [num_pages, 64, D] and
    block_table [B, Hkv, C // 64] int32 maps each unit's 64-slot pages into them."""
    K: torch.Tensor
    V: torch.Tensor
    pos: torch.Tensor
    n: torch.Tensor
    seqlen: torch.Tensor
    block_table: Optional[torch.Tensor] = None

    @property
    def B(self): return self.pos.shape[0]

    @property
    def Hkv(self): return self.pos.shape[1]

    @property
    def C(self): return self.pos.shape[2]

    @property
    def D(self): return self.K.shape[-1]

    @property
    def num_pages(self): return self.K.shape[0] if self.block_table is not None else 0

    @classmethod
    def empty(cls, B, Hkv, C_, D, device="cuda"):
        return cls(K=torch.zeros(B, Hkv, C_, D, dtype=torch.float16, device=device),
                   V=torch.zeros(B, Hkv, C_, D, dtype=torch.float16, device=device),
                   pos=torch.full((B, Hkv, C_), -1, dtype=torch.int32, device=device),
                   n=torch.zeros(B, Hkv, dtype=torch.int32, device=device),
                   seqlen=torch.zeros(B, dtype=torch.int32, device=device))

    @classmethod
    def empty_paged(cls, B, Hkv, C_, D, num_pages, block_table=None, device="cuda"):
        """Paged cache: pools of num_pages pages of 64 slots; block_table [B, Hkv, C_ // 64]
        (default: unit u owns pages u * C_ / 64 .. (u + 1) * C_ / 64 - 1)."""
        if C_ % PAGE_SLOTS:
            raise ValueError("C must be a multiple of 64 in the paged layout")
        if block_table is None:
            block_table = torch.arange(B * Hkv * (C_ // PAGE_SLOTS), dtype=torch.int32,
                                       device=device).view(B, Hkv, C_ // PAGE_SLOTS)
        return cls(K=torch.zeros(num_pages, PAGE_SLOTS, D, dtype=torch.float16, device=device),
                   V=torch.zeros(num_pages, PAGE_SLOTS, D, dtype=torch.float16, device=device),
                   pos=torch.full((B, Hkv, C_), -1, dtype=torch.int32, device=device),
                   n=torch.zeros(B, Hkv, dtype=torch.int32, device=device),
                   seqlen=torch.zeros(B, dtype=torch.int32, device=device),
                   block_table=block_table.to(device=device, dtype=torch.int32).contiguous())

    def __getstate__(self):
        return _state_without_desc(self)

    def desc(self) -> SlotCacheDesc:
        # built once and kept while the fields' storage, shapes and strides stay the same (a
        # field replaced or resized in place yields a new key, and the fields are checked again)
        t = (self.K, self.V, self.pos, self.n, self.seqlen, self.block_table)
        key = _desc_key(t)
        d = self.__dict__.get("_desc")
        if d is not None and self.__dict__.get("_desc_key") == key:
            return d
        d = SlotCacheDesc(self.B, self.Hkv, self.D, self.C, _ptr(self.K), _ptr(self.V),
                          _ptr(self.pos), _ptr(self.n), _ptr(self.seqlen),
                          _ptr(self.block_table), self.num_pages)
        self.__dict__["_desc"], self.__dict__["_desc_key"] = d, key
        self.__dict__["_desc_p"] = C.pointer(d)
        return d


@dataclass
class QuantCache:
    """KIVI cache in device memory (layout documented in include/kvc.h).  Dense layout:
    k_blocks, v_blocks [B, Hkv, Cq / 32, block_bytes].  Paged layout: pools
    [num_pages, 4, block_bytes] of 4-group (128-token) pages, block_table [B, Hkv, Cq / 128]."""
    k_blocks: torch.Tensor
    v_blocks: torch.Tensor
    k_res: torch.Tensor
    v_res: torch.Tensor
    len: torch.Tensor
    bits: int
    R: int
    block_table: Optional[torch.Tensor] = None
    Cq_paged: int = 0
    k_gear: Optional[torch.Tensor] = None   # GEAR side blocks [B, Hkv, Cq / 32, side_bytes]
    v_gear: Optional[torch.Tensor] = None

    @property
    def B(self): return self.k_res.shape[0]

    @property
    def Hkv(self): return self.k_res.shape[1]

    @property
    def D(self): return self.k_res.shape[3]

    @property
    def Cq(self):
        return self.Cq_paged if self.block_table is not None else self.k_blocks.shape[2] * KIVI_GROUP

    @property
    def num_pages(self): return self.k_blocks.shape[0] if self.block_table is not None else 0

    @classmethod
    def empty(cls, B, Hkv, Cq, D, bits, R, device="cuda", gear=False):
        """KIVI cache; gear=True adds the GEAR side blocks (sparse + rank-2 corrections)."""
        assert Cq % KIVI_GROUP == 0
        bb = KIVI_GROUP * D * bits // 8 + 4 * D
        ng = Cq // KIVI_GROUP
        sb = kvc_gear_side_bytes(D) if gear else 0
        return cls(k_blocks=torch.zeros(B, Hkv, ng, bb, dtype=torch.uint8, device=device),
                   v_blocks=torch.zeros(B, Hkv, ng, bb, dtype=torch.uint8, device=device),
                   k_res=torch.zeros(B, Hkv, R + KIVI_GROUP, D, dtype=torch.float16, device=device),
                   v_res=torch.zeros(B, Hkv, R + KIVI_GROUP, D, dtype=torch.float16, device=device),
                   len=torch.zeros(B, dtype=torch.int32, device=device), bits=bits, R=R,
                   k_gear=torch.zeros(B, Hkv, ng, sb, dtype=torch.uint8, device=device)
                   if gear else None,
                   v_gear=torch.zeros(B, Hkv, ng, sb, dtype=torch.uint8, device=device)
                   if gear else None)

    @classmethod
    def empty_paged(cls, B, Hkv, Cq, D, bits, R, num_pages, block_table=None, device="cuda",
                    gear=False):
        """Paged KIVI cache: pools of num_pages pages of 4 groups; block_table [B, Hkv, Cq / 128]
        (default: unit u owns pages u * Cq / 128 .. (u + 1) * Cq / 128 - 1).  gear=True adds
        GEAR side-block pools [num_pages, 4, side_bytes] behind the same table."""
        page = KIVI_GROUP * KIVI_PAGE_GROUPS
        if Cq % page:
            raise ValueError("Cq must be a multiple of 128 in the paged layout")
        if block_table is None:
            block_table = torch.arange(B * Hkv * (Cq // page), dtype=torch.int32,
                                       device=device).view(B, Hkv, Cq // page)
        bb = KIVI_GROUP * D * bits // 8 + 4 * D
        pool = (num_pages, KIVI_PAGE_GROUPS, bb)
        side = (num_pages, KIVI_PAGE_GROUPS, kvc_gear_side_bytes(D))
        return cls(k_blocks=torch.zeros(pool, dtype=torch.uint8, device=device),
                   v_blocks=torch.zeros(pool, dtype=torch.uint8, device=device),
                   k_res=torch.zeros(B, Hkv, R + KIVI_GROUP, D, dtype=torch.float16, device=device),
                   v_res=torch.zeros(B, Hkv, R + KIVI_GROUP, D, dtype=torch.float16, device=device),
                   len=torch.zeros(B, dtype=torch.int32, device=device), bits=bits, R=R,
                   block_table=block_table.to(device=device, dtype=torch.int32).contiguous(),
                   Cq_paged=Cq,
                   k_gear=torch.zeros(side, dtype=torch.uint8, device=device) if gear else None,
                   v_gear=torch.zeros(side, dtype=torch.uint8, device=device) if gear else None)

    def __getstate__(self):
        return _state_without_desc(self)

    def desc(self) -> QuantCacheDesc:
        # kept while the fields' storage, shapes and strides stay the same (see SlotCache)
        t = (self.k_blocks, self.v_blocks, self.k_res, self.v_res, self.len, self.block_table,
             self.k_gear, self.v_gear)
        key = _desc_key(t) + (self.bits, self.R, self.Cq_paged)
        d = self.__dict__.get("_desc")
        if d is not None and self.__dict__.get("_desc_key") == key:
            return d
        d = QuantCacheDesc(self.B, self.Hkv, self.D, self.bits, self.R, self.Cq,
                           _ptr(self.k_blocks), _ptr(self.v_blocks), _ptr(self.k_res),
                           _ptr(self.v_res), _ptr(self.len), _ptr(self.block_table),
                           self.num_pages, _ptr(self.k_gear), _ptr(self.v_gear))
        self.__dict__["_desc"], self.__dict__["_desc_key"] = d, key
        self.__dict__["_desc_p"] = C.pointer(d)
        return d
