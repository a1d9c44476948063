"""GEAR-4 oracle -- TEST INFRASTRUCTURE ONLY (same rules as the rest of ``oracle``).

GEAR ("Rethinking KV Cache Compression" guide, §2: GEAR sparsity 2%, rank 2; §16 "前置背景、
复现方法与结论边界": on top of KIVI's quantisation residual GEAR adds a 2% sparse and a rank-2
low-rank correction) compresses every flushed 32-token group of K and of V as
    X  ~  Xq + S + L
  Xq  the KIVI quantisation of the group (codes, scales and zeros exactly as ``kivi_quantize_unit``)
  E   the quantisation residual, defined in fp32: xq = fl32(zero + code * scale) (one rounding),
      e = fl32(x - xq)
  S   the ceil(2% * 32 * D) entries of E with the largest |e| (ties: lower flat index t * D + d),
      stored as their flat index and binary16 value RN16(e)
  L   the best rank-2 approximation (truncated SVD) of R = E with the S entries set to zero,
      stored as A [2, 32] (orthonormal left factors) and B [2, D] = A R, both binary16
and decode attention runs over the reconstruction  x_hat = xq + S + L  (exact fp64 here; the
fp16 residual ring of the newest tokens is used as is, as for KIVI).

Everything is fp64 except the residual, which is fp32 by definition so that the sparse selection
(an integer decision) is made in the same precision on both sides.  numpy.linalg.svd provides
the truncated SVD.  Pinned in tests/test_oracle_gear.py.
"""
from __future__ import annotations

import math

import numpy as np

from . import G_KIVI, kivi_nq, kivi_quantize_unit

GEAR_SPARSITY_PCT = 2   # percent of a group's entries kept exactly
GEAR_RANK = 2


def n_sparse(D: int, G: int = G_KIVI, pct: int = GEAR_SPARSITY_PCT) -> int:
    """Entries of a G x D group kept in the sparse part: ceil(pct% * G * D)."""
    return (pct * G * D + 99) // 100


def side_bytes(D: int, G: int = G_KIVI) -> int:
    """Bytes of one group's GEAR side data: n_s u16 indices, n_s binary16 values, A [2, G] and
    B [2, D] binary16, padded to 16 bytes."""
    raw = 4 * n_sparse(D, G) + 2 * GEAR_RANK * G + 2 * GEAR_RANK * D
    return (raw + 15) // 16 * 16


def _f16(bits) -> np.ndarray:
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _dequant_f32(codes, scale_bits, zero_bits) -> np.ndarray:
    """xq = fl32(zero + code * scale): the exact value (fp64 holds it) rounded once to fp32."""
    return (_f16(zero_bits) + codes.astype(np.float64) * _f16(scale_bits)).astype(np.float32)


def group_parts(x16, codes, scale_bits, zero_bits, pct: int = GEAR_SPARSITY_PCT,
                rank: int = GEAR_RANK) -> dict:
    """GEAR parts of one group: x16 [G, D] binary16 values, codes [G, D], and the per-element
    scale / zero bit patterns [G, D] of their KIVI quantisation.  Returns the fp32 residual E,
    the sparse flat indices (ascending) and their binary16 values, R, and the truncated SVD
    factors A [rank, G] (orthonormal rows) and B [rank, D] = A R (fp64)."""
    G, D = x16.shape
    xq = _dequant_f32(codes, scale_bits, zero_bits)
    E = (np.asarray(x16, np.float16).astype(np.float32) - xq).astype(np.float32)
    flat = np.abs(E).reshape(-1)
    ns = n_sparse(D, G, pct)
    # largest |e| first, ties to the lower flat index
    order = np.lexsort((np.arange(flat.size), -flat.astype(np.float64)))
    idx = np.sort(order[:ns])
    vals = E.reshape(-1)[idx].astype(np.float16)
    R = E.astype(np.float64).reshape(-1).copy()
    R[idx] = 0.0
    R = R.reshape(G, D)
    if rank > 0:
        U, s, Vt = np.linalg.svd(R, full_matrices=False)
        A = U[:, :rank].T.copy()
        B = A @ R
    else:
        A = np.zeros((0, G))
        B = np.zeros((0, D))
    return {"E": E, "idx": idx.astype(np.uint16), "val": vals, "R": R, "A": A, "B": B,
            "xq": xq}


def _expand_params(qz, n_q: int, D: int, G: int = G_KIVI):
    """Per-element scale / zero bit patterns [n_q, D] of K (per channel per group) and V (per
    token per channel group) from a ``kivi_quantize_unit`` result."""
    ks = np.repeat(qz["k_scale"], G, axis=0)[:n_q]
    kz = np.repeat(qz["k_zero"], G, axis=0)[:n_q]
    vs = np.repeat(qz["v_scale"], G, axis=1)
    vz = np.repeat(qz["v_zero"], G, axis=1)
    return ks, kz, vs, vz


def quantize_unit(K, V, n_q: int, bits: int = 4, pct: int = GEAR_SPARSITY_PCT,
                  rank: int = GEAR_RANK, G: int = G_KIVI) -> dict:
    """GEAR compression of one unit's first n_q tokens.  Returns the KIVI result ``qz`` plus,
    per group g, ``k[g]`` / ``v[g]`` = ``group_parts`` of its K and V."""
    K16 = np.asarray(K, np.float16)
    V16 = np.asarray(V, np.float16)
    D = K16.shape[1]
    qz = kivi_quantize_unit(K16, V16, n_q, bits, G)
    ks, kz, vs, vz = _expand_params(qz, n_q, D, G)
    out = {"qz": qz, "k": [], "v": [], "bits": bits}
    for g in range(n_q // G):
        sl = slice(g * G, (g + 1) * G)
        out["k"].append(group_parts(K16[sl], qz["k_codes"][sl], ks[sl], kz[sl], pct, rank))
        out["v"].append(group_parts(V16[sl], qz["v_codes"][sl], vs[sl], vz[sl], pct, rank))
    return out


def reconstruct(parts: dict, half_factors: bool = True) -> np.ndarray:
    """x_hat = xq + S + L of one group in fp64: S from the stored binary16 values, L = A^T B from
    the factors (rounded to binary16 first when half_factors, as they are stored)."""
    G, D = parts["E"].shape
    x = parts["xq"].astype(np.float64).reshape(-1).copy()
    x[parts["idx"].astype(np.int64)] += parts["val"].astype(np.float64)
    x = x.reshape(G, D)
    A, B = parts["A"], parts["B"]
    if half_factors:
        A = A.astype(np.float16).astype(np.float64)
        B = B.astype(np.float16).astype(np.float64)
    return x + A.T @ B


def attend_unit(q, K, V, T: int, R: int, bits: int = 4, gz: dict | None = None,
                scale: float | None = None, pct: int = GEAR_SPARSITY_PCT, rank: int = GEAR_RANK,
                G: int = G_KIVI):
    """GEAR decode attention for one unit: full softmax attention (fp64) of q [g, D] over the
    reconstructed tokens [0, n_q) and the raw binary16 tokens [n_q, T).  Returns (out, lse)."""
    q = np.asarray(q, np.float16).astype(np.float64)
    K16 = np.asarray(K, np.float16)
    V16 = np.asarray(V, np.float16)
    D = K16.shape[1]
    n_q = kivi_nq(T, R, G)
    if gz is None:
        gz = quantize_unit(K16[:n_q], V16[:n_q], n_q, bits, pct, rank, G)
    Kh = np.concatenate([reconstruct(p) for p in gz["k"]] +
                        [K16[n_q:T].astype(np.float64)]) if T else np.zeros((0, D))
    Vh = np.concatenate([reconstruct(p) for p in gz["v"]] +
                        [V16[n_q:T].astype(np.float64)]) if T else np.zeros((0, D))
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    s = scale * (q @ Kh.T)                       # [g, T]
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    l = w.sum(axis=1, keepdims=True)
    return (w @ Vh) / l, (m + np.log(l))[:, 0]


def pack_side(parts: dict, D: int, G: int = G_KIVI) -> np.ndarray:
    """One group's side block: n_s u16 indices, n_s binary16 values, A [2, G], B [2, D]
    (binary16, row-major), zero padding to side_bytes(D)."""
    out = np.zeros(side_bytes(D, G), np.uint8)
    ns = n_sparse(D, G)
    raw = np.concatenate([parts["idx"].astype(np.uint16).view(np.uint8),
                          parts["val"].astype(np.float16).view(np.uint8),
                          parts["A"].astype(np.float16).reshape(-1).view(np.uint8),
                          parts["B"].astype(np.float16).reshape(-1).view(np.uint8)])
    assert raw.size == 4 * ns + 4 * G + 4 * D
    out[:raw.size] = raw
    return out
