"""Seeded synthetic workloads for the compressed-KV decode path.

This module holds shapes and seeded input generators only -- none of the
method's arithmetic.  It is the one module the tests, the benchmark and the
oracle-side checks share: every input is drawn here from a seed, in fp32 from a
``torch.Generator`` and rounded to binary16 (round-to-nearest-even), so both
sides of a parity check see the same bit patterns.

The five workloads restate the shapes the pages' experiments use (LLaMA-7B and
LLaMA3-70B / Qwen3-32B shaped layers, KIVI G=32 / R=128, StreamingLLM and H2O
budgets of 64 + 448, random eviction with the prompt locked).  The pages'
datasets (ShareGPT, LongBench, LiveCodeBench traces) and model weights are not
available; these synthetic caches stand in for their shapes only.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    T: int                      # tokens in the cache at the decode step (incl. current)
    seed: int
    methods: tuple = ()
    n_sink: int = 0             # StreamingLLM sinks
    n_recent: int = 0           # StreamingLLM / H2O recent window
    n_heavy: int = 0            # H2O heavy hitters
    kivi_bits: tuple = ()
    kivi_R: int = 128
    prompt_len: int = 0         # random eviction: locked prompt
    keep_ratio: float = 0.0
    evict_every: int = 0
    decode_steps: int = 0
    outlier_frac: float = 0.0   # fraction of channels scaled x10 in K and V (per KV head)
    offset_range: float = 0.0   # per-(head, channel) offsets U(-a, a) added to Q, K, V
    notes: str = ""
    extra: dict = field(default_factory=dict)


TINY = Workload(
    name="tiny-mha4-d64", B=1, Hq=4, Hkv=4, D=64, T=96, seed=1001,
    methods=("fp16", "stream", "h2o", "kivi4", "random"),
    n_sink=4, n_recent=12, n_heavy=8, kivi_bits=(4,), kivi_R=16, prompt_len=16, keep_ratio=0.5,
    decode_steps=32, notes="prompt 64 tokens then 32 decode steps; H2O 8 heavy + 8 recent",
    extra={"prompt": 64, "h2o_recent": 8})

LLAMA7B = Workload(
    name="llama7b-b8-h32-d128-t2048", B=8, Hq=32, Hkv=32, D=128, T=2048, seed=1002,
    methods=("fp16", "stream", "h2o"), n_sink=64, n_recent=448, n_heavy=64,
    outlier_frac=0.02, notes="3 outlier channels x10 per KV head in K and V; H2O prefill "
    "scores from a 2048-token causal prompt")

KIVI_MHA = Workload(
    name="kivi-b32-h32-d128-t4096", B=32, Hq=32, Hkv=32, D=128, T=4096, seed=1003,
    methods=("fp16", "kivi2", "kivi4"), kivi_bits=(2, 4), kivi_R=128, offset_range=2.0,
    notes="N(0,1) plus per-(head, channel) offsets U(-2,2) on Q, K, V")

HEAVY = Workload(
    name="heavy-gqa64x8-b512-d128-t2048", B=512, Hq=64, Hkv=8, D=128, T=2048, seed=1004,
    methods=("fp16", "h2o", "kivi4", "stream"), n_sink=64, n_recent=448, n_heavy=64,
    kivi_bits=(4,), kivi_R=128,
    notes="LLaMA3-70B-shaped layer; one decode step per method; H2O prefill score pass over "
    "the 2048-token prompt")

REASONING = Workload(
    name="reasoning-gqa64x8-b16-d128-t32768", B=16, Hq=64, Hkv=8, D=128, T=32768, seed=1005,
    methods=("fp16", "random"), prompt_len=1024, keep_ratio=0.25, evict_every=1024,
    notes="Qwen3-32B-shaped layer; evict every 1024 generated tokens to keep 0.25 per KV head")

WORKLOADS = {w.name: w for w in (TINY, LLAMA7B, KIVI_MHA, HEAVY, REASONING)}

# Seed of the random-eviction Philox key (the hexadecimal digits of pi).
RANDOM_EVICT_SEED = 0x243F6A8885A308D3


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_f16(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """N(0,1) drawn in fp32 and rounded to binary16."""
    return torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32).half()


def outlier_channels(Hkv: int, D: int, frac: float, gen: torch.Generator) -> torch.Tensor:
    """Per KV head, round(frac * D) distinct channels -> bool mask [Hkv, D]."""
    k = int(round(frac * D))
    mask = torch.zeros(Hkv, D, dtype=torch.bool)
    for h in range(Hkv):
        idx = torch.randperm(D, generator=gen)[:k]
        mask[h, idx] = True
    return mask


def kv_tensors(w: Workload, T: int | None = None, B: int | None = None, device="cpu",
               seed_offset: int = 0):
    """K, V [B, Hkv, T, D] binary16 for workload w (with its outliers / offsets)."""
    T = w.T if T is None else T
    B = w.B if B is None else B
    gen = generator(w.seed + seed_offset, device)
    K = normal_f16((B, w.Hkv, T, w.D), gen, device)
    V = normal_f16((B, w.Hkv, T, w.D), gen, device)
    cpu_gen = generator(w.seed + 7777 + seed_offset)
    if w.outlier_frac > 0:
        mask = outlier_channels(w.Hkv, w.D, w.outlier_frac, cpu_gen).to(device)
        scale = torch.where(mask, torch.tensor(10.0, device=device), torch.tensor(1.0, device=device))
        K = (K.float() * scale[None, :, None, :]).half()
        V = (V.float() * scale[None, :, None, :]).half()
    if w.offset_range > 0:
        offk = (torch.rand(w.Hkv, w.D, generator=cpu_gen) * 2 - 1) * w.offset_range
        offv = (torch.rand(w.Hkv, w.D, generator=cpu_gen) * 2 - 1) * w.offset_range
        K = (K.float() + offk.to(device)[None, :, None, :]).half()
        V = (V.float() + offv.to(device)[None, :, None, :]).half()
    return K, V


def q_tensor(w: Workload, B: int | None = None, device="cpu", seed_offset: int = 0, L: int = 1):
    """Decode queries [B, Hq, D] (L == 1) or prompt queries [B, Hq, L, D], binary16."""
    B = w.B if B is None else B
    gen = generator(w.seed + 100 + seed_offset, device)
    shape = (B, w.Hq, w.D) if L == 1 else (B, w.Hq, L, w.D)
    Q = normal_f16(shape, gen, device)
    if w.offset_range > 0:
        cpu_gen = generator(w.seed + 8888)
        offq = (torch.rand(w.Hq, w.D, generator=cpu_gen) * 2 - 1) * w.offset_range
        offq = offq.to(device)
        Q = (Q.float() + (offq[None] if L == 1 else offq[None, :, None, :])).half()
    return Q


def new_token_kv(w: Workload, step: int, B: int | None = None, device="cpu"):
    """The K/V of one generated token per sequence, [B, Hkv, 1, D] each."""
    B = w.B if B is None else B
    gen = generator(w.seed + 5000 + step, device)
    return (normal_f16((B, w.Hkv, 1, w.D), gen, device),
            normal_f16((B, w.Hkv, 1, w.D), gen, device))
