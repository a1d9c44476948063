"""fp64 CPU oracle for the compressed-KV decode path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it; the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64, libm); this module only
marshals numpy arrays.  Inputs are binary16 bit patterns (``np.float16`` arrays
are viewed as ``uint16``).  Every function states the passage it follows.

Parity unpinned: none of the functions below lacks an independent pin; see the
``tests/test_oracle_*.py`` files for what pins each one.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

G_KIVI = 32  # KIVI group size fixed by the pages (Rethinking KV Cache Compression, §2)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (IEEE semantics, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = C.CDLL(_LIB_PATH)
            P = C.c_void_p
            i, l, d, u32, u64 = C.c_int, C.c_long, C.c_double, C.c_uint32, C.c_uint64
            sig = {
                "orc_half_to_double": (d, [C.c_uint16]),
                "orc_double_to_half": (C.c_uint16, [d]),
                "orc_half_to_double_array": (None, [l, P, P]),
                "orc_double_to_half_array": (None, [l, P, P]),
                "orc_decode_attend": (None, [i, i, i, i, i, P, P, P, P, d, P, P, P, i]),
                "orc_kivi_nq": (l, [l, i, i]),
                "orc_kivi_quantize_unit": (None, [i, i, i, l, P, P, P, P, P, P, P, P]),
                "orc_kivi_pack_group": (None, [i, i, i, P, P, P, P, P, P, P, P]),
                "orc_kivi_attend_unit": (None, [i, i, i, l, l, P, P, P, P, P, P, P, P, P, d, P, P]),
                "orc_h2o_prefill_scores": (None, [i, i, i, i, i, l, l, P, P, d, P, i]),
                "orc_h2o_accumulate": (None, [i, i, i, i, P, P, P, C.c_double, P]),
                "orc_h2o_keep": (i, [i, P, P, l, i, i, P, P]),
                "orc_stream_keep": (i, [i, P, l, i, i, P]),
                "orc_philox4x32_10": (None, [P, P, P]),
                "orc_random_key": (u64, [u64, C.c_int32, i, i, u32]),
                "orc_random_keep": (i, [i, P, i, d, u64, u32, i, i, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected float16/uint16 array, got {a.dtype}")
    return np.ascontiguousarray(a)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# --------------------------------------------------------------------------- binary16

def half_to_double(bits) -> np.ndarray:
    """Exact widening of binary16 bit patterns to fp64 (IEEE 754 binary16 definition)."""
    b = _u16(bits)
    out = np.empty(b.shape, np.float64)
    _L().orc_half_to_double_array(b.size, _ptr(b), _ptr(out))
    return out


def double_to_half(x) -> np.ndarray:
    """Round-to-nearest-even narrowing of fp64 values to binary16 bit patterns."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, np.uint16)
    _L().orc_double_to_half_array(x.size, _ptr(x), _ptr(out))
    return out


# --------------------------------------------------------------------------- attention

def decode_attend(q, K, V, n, scale: float | None = None, want_logits: bool = False,
                  threads: int = 1):
    """Full softmax attention of every query head over the valid slots of its KV head.

    q [B,Hq,D], K/V [B,Hkv,C,D] (binary16), n [B,Hkv] valid slots.  Query head h
    reads KV head h // (Hq // Hkv).  Returns (out [B,Hq,D] f64, lse [B,Hq] f64,
    logits [B,Hq,C] f64 or None).  Scaled dot-product attention with scale 1/sqrt(D).
    """
    q, K, V = _u16(q), _u16(K), _u16(V)
    B, Hq, D = q.shape
    _, Hkv, Cc, D2 = K.shape
    assert D2 == D and V.shape == K.shape and Hq % Hkv == 0
    n = _i32(n).reshape(B, Hkv)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    logits = np.full((B, Hq, Cc), np.nan, np.float64) if want_logits else None
    _L().orc_decode_attend(B, Hq, Hkv, D, Cc, _ptr(q), _ptr(K), _ptr(V), _ptr(n), float(scale),
                           _ptr(out), _ptr(lse), _ptr(logits) if want_logits else None,
                           int(threads))
    return out, lse, logits


# --------------------------------------------------------------------------- KIVI

def kivi_nq(T: int, R: int, G: int = G_KIVI) -> int:
    """Tokens held quantised for a sequence of T tokens: G * floor(max(0, T - R) / G)."""
    return int(_L().orc_kivi_nq(int(T), int(G), int(R)))


def kivi_quantize_unit(K, V, n_q: int, bits: int, G: int = G_KIVI) -> dict:
    """KIVI quantisation of one unit's first n_q tokens (K per channel, V per token).

    K, V [T,D] binary16.  Returns logical codes (one per element), scale and zero
    bit patterns: k_scale/k_zero [n_q/G, D], v_scale/v_zero [n_q, D/G].
    """
    K, V = _u16(K), _u16(V)
    T, D = K.shape
    assert n_q % G == 0 and n_q <= T and D % G == 0
    ng = n_q // G
    r = {
        "k_scale": np.zeros((ng, D), np.uint16), "k_zero": np.zeros((ng, D), np.uint16),
        "k_codes": np.zeros((n_q, D), np.uint8),
        "v_scale": np.zeros((n_q, D // G), np.uint16), "v_zero": np.zeros((n_q, D // G), np.uint16),
        "v_codes": np.zeros((n_q, D), np.uint8),
    }
    _L().orc_kivi_quantize_unit(D, G, bits, n_q, _ptr(K), _ptr(V), _ptr(r["k_scale"]),
                                _ptr(r["k_zero"]), _ptr(r["k_codes"]), _ptr(r["v_scale"]),
                                _ptr(r["v_zero"]), _ptr(r["v_codes"]))
    return r


def kivi_block_bytes(D: int, bits: int, G: int = G_KIVI) -> int:
    """Bytes of one packed K (or V) group block: G*D*bits/8 code bytes + 4*D bytes of scale/zero."""
    return G * D * bits // 8 + 4 * D


def kivi_pack_unit(qz: dict, D: int, bits: int, G: int = G_KIVI):
    """Pack every group of a unit into the documented K/V block layout -> (k_blocks, v_blocks) u8."""
    ng = qz["k_scale"].shape[0]
    bb = kivi_block_bytes(D, bits, G)
    kb = np.zeros((ng, bb), np.uint8)
    vb = np.zeros((ng, bb), np.uint8)
    for g in range(ng):
        kc = np.ascontiguousarray(qz["k_codes"][g * G:(g + 1) * G])
        vc = np.ascontiguousarray(qz["v_codes"][g * G:(g + 1) * G])
        ks = np.ascontiguousarray(qz["k_scale"][g]); kz = np.ascontiguousarray(qz["k_zero"][g])
        vs = np.ascontiguousarray(qz["v_scale"][g * G:(g + 1) * G])
        vz = np.ascontiguousarray(qz["v_zero"][g * G:(g + 1) * G])
        kbg = np.zeros(bb, np.uint8); vbg = np.zeros(bb, np.uint8)
        _L().orc_kivi_pack_group(D, G, bits, _ptr(kc), _ptr(ks), _ptr(kz), _ptr(vc), _ptr(vs),
                                 _ptr(vz), _ptr(kbg), _ptr(vbg))
        kb[g] = kbg; vb[g] = vbg
    return kb, vb


def kivi_attend_unit(q, K, V, T: int, R: int, bits: int, qz: dict | None = None,
                     scale: float | None = None, G: int = G_KIVI):
    """KIVI decode attention for one unit: exact dequantised tokens [0,n_q) + fp16 residual.

    q [g,D]; K, V [>=T, D] raw binary16 tokens of the unit.  Returns (out [g,D], lse [g]).
    """
    q, K, V = _u16(q), _u16(K), _u16(V)
    g, D = q.shape
    n_q = kivi_nq(T, R, G)
    if qz is None:
        qz = kivi_quantize_unit(K[:T], V[:T], n_q, bits, G)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((g, D), np.float64)
    lse = np.zeros(g, np.float64)
    Kc = np.ascontiguousarray(K[:T]); Vc = np.ascontiguousarray(V[:T])
    _L().orc_kivi_attend_unit(g, D, G, T, n_q, _ptr(q), _ptr(Kc), _ptr(Vc), _ptr(qz["k_scale"]),
                              _ptr(qz["k_zero"]), _ptr(qz["k_codes"]), _ptr(qz["v_scale"]),
                              _ptr(qz["v_zero"]), _ptr(qz["v_codes"]), float(scale), _ptr(out),
                              _ptr(lse))
    return out, lse


# --------------------------------------------------------------------------- H2O

def h2o_prefill_scores(Qp, Kp, L: int, scale: float | None = None, threads: int = 1,
                       score_cap: int | None = None):
    """Heavy-hitter scores over a causal prompt: column sums of the softmax rows, summed
    over each KV head's query group.  Qp [B,Hq,L,D], Kp [B,Hkv,cap,D] -> [B,Hkv,score_cap]."""
    Qp, Kp = _u16(Qp), _u16(Kp)
    B, Hq, L2, D = Qp.shape
    _, Hkv, cap, _ = Kp.shape
    assert L2 == L and cap >= L
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    sc = score_cap or L
    scores = np.zeros((B, Hkv, sc), np.float64)
    _L().orc_h2o_prefill_scores(B, Hq, Hkv, D, L, cap, sc, _ptr(Qp), _ptr(Kp), float(scale),
                                _ptr(scores), int(threads))
    return scores


def h2o_accumulate(scores, logits, lse, n, decay: float = 0.0):
    """p[b,hk,j] = sum_{h in group(hk)} exp(logits[b,h,j] - lse[b,h]) for j < n[b,hk];
    decay 0: scores += p; decay in (0, 1): scores = decay * scores + (1 - decay) * p."""
    scores = np.ascontiguousarray(np.array(scores, dtype=np.float64))
    logits = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    lse = np.ascontiguousarray(np.asarray(lse, dtype=np.float64))
    B, Hkv, Cc = scores.shape
    Hq = logits.shape[1]
    n = _i32(n).reshape(B, Hkv)
    _L().orc_h2o_accumulate(B, Hq, Hkv, Cc, _ptr(n), _ptr(logits), _ptr(lse), float(decay),
                            _ptr(scores))
    return scores


def h2o_keep(pos, score, T: int, n_heavy: int, n_recent: int):
    """H2O keep-set of one unit's n slots -> (keep mask bool [n], relative margin)."""
    pos = _i32(pos)
    score = np.ascontiguousarray(np.asarray(score, dtype=np.float64))
    n = pos.size
    keep = np.zeros(n, np.uint8)
    margin = C.c_double(0.0)
    _L().orc_h2o_keep(n, _ptr(pos), _ptr(score), int(T), int(n_heavy), int(n_recent), _ptr(keep),
                      C.byref(margin))
    return keep.astype(bool), margin.value


# --------------------------------------------------------------------------- StreamingLLM

def stream_keep(pos, T: int, n_sink: int, n_recent: int):
    """StreamingLLM keep mask: position < n_sink or position >= T - n_recent."""
    pos = _i32(pos)
    keep = np.zeros(pos.size, np.uint8)
    _L().orc_stream_keep(pos.size, _ptr(pos), int(T), int(n_sink), int(n_recent), _ptr(keep))
    return keep.astype(bool)


# --------------------------------------------------------------------------- random eviction

def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 block: 4 x u32 counter, 2 x u32 key -> 4 x u32 (Salmon et al., SC'11)."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    o = np.zeros(4, np.uint32)
    _L().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(o))
    return o


def random_key(seed: int, pos: int, kv_head: int, batch: int, epoch: int) -> int:
    """64-bit eviction key (Philox out[0] << 32 | out[1]) with counter (pos, kv_head, batch, epoch)."""
    return int(_L().orc_random_key(seed & (2**64 - 1), int(pos), int(kv_head), int(batch),
                                   epoch & 0xffffffff))


def random_keep(pos, prompt_len: int, keep_ratio: float, seed: int, epoch: int, batch: int,
                kv_head: int):
    """Per-head random eviction keep mask for one unit (prompt locked, n_keep smallest keys)."""
    pos = _i32(pos)
    keep = np.zeros(pos.size, np.uint8)
    _L().orc_random_keep(pos.size, _ptr(pos), int(prompt_len), float(keep_ratio),
                         seed & (2**64 - 1), epoch & 0xffffffff, int(batch), int(kv_head),
                         _ptr(keep))
    return keep.astype(bool)


def n_keep_of(n_cand: int, keep_ratio: float) -> int:
    """n_keep = max(1, int(n_cand * keep_ratio)) for n_cand > 0 (the pages' formula)."""
    return max(1, int(n_cand * keep_ratio)) if n_cand > 0 else 0
