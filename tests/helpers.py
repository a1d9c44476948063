"""Shared test helpers: tolerances and tensor <-> numpy marshalling (no method arithmetic)."""
import numpy as np
import torch

# Attention outputs are fp16.  The stated bound is 2e-3 absolute; the output is
# additionally rounded to binary16, so half an fp16 ulp of the reference value
# is added (it exceeds 2e-3 only for |o| >= 8).
O_ABS_TOL = 2e-3
# Accumulated H2O scores: 1e-4 relative.
SCORE_REL_TOL = 1e-4
# Log-sum-exp and logits are fp32 values compared against fp64.
LSE_ABS_TOL = 1e-4


def o_tolerance(ref: np.ndarray) -> np.ndarray:
    r16 = np.abs(ref).astype(np.float16)
    return O_ABS_TOL + np.spacing(r16).astype(np.float64) / 2


def assert_o_close(o_gpu, ref, what="o"):
    o = np.asarray(o_gpu, dtype=np.float64)
    err = np.abs(o - ref)
    tol = o_tolerance(ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def np16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.float16)


def slot_cache_from(kvc, K: torch.Tensor, V: torch.Tensor, n, C: int, seqlen=None):
    """A slot cache whose unit (b, h) holds tokens 0..n[b,h]-1 of K/V [B,Hkv,T,D] in slots 0..n-1."""
    B, Hkv, T, D = K.shape
    cache = kvc.SlotCache.empty(B, Hkv, C, D, device="cuda")
    m = min(T, C)
    cache.K[:, :, :m] = K[:, :, :m].cuda()
    cache.V[:, :, :m] = V[:, :, :m].cuda()
    cache.pos[:, :, :C] = torch.arange(C, dtype=torch.int32, device="cuda")
    n = torch.as_tensor(np.asarray(n, dtype=np.int32)).reshape(B, Hkv)
    cache.n.copy_(n.cuda())
    sl = n.max(1).values if seqlen is None else torch.as_tensor(seqlen, dtype=torch.int32)
    cache.seqlen.copy_(sl.to(torch.int32).cuda())
    return cache


def device_status_clean(kvc):
    torch.cuda.synchronize()
    return kvc.kvc_read_device_status() == 0
