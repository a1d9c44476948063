"""The oracle's Philox4x32-10 against a second library implementation: cuRAND's
Philox4_32_10 device generator, built from tests/pins/curand_philox.cu and run
on the GPU (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11,
defines the block function both implement)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.gpu
def test_philox_matches_curand(orc, tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = tmp_path / "curand_philox"
    subprocess.run([nvcc, "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
                    os.path.join(HERE, "pins", "curand_philox.cu"), "-o", str(exe)],
                   check=True, capture_output=True, timeout=600)
    rng = np.random.default_rng(11)
    seeds = [int(x) for x in rng.integers(0, 2**63, 60, dtype=np.uint64)] + [0, 2**64 - 1, 1, 2**32]
    subs = [int(x) for x in rng.integers(0, 2**63, 60, dtype=np.uint64)] + [0, 2**64 - 1, 2**32 - 1, 5]
    ctrs = [int(x) for x in rng.integers(0, 2**62, 60, dtype=np.uint64)] + [0, 2**62 - 1, 2**32, 7]
    # the counter words the eviction keys use: (pos, kv_head, batch, epoch)
    for pos, hk, b, ep in [(0, 0, 0, 0), (1023, 7, 15, 31), (32767, 3, 2, 1)]:
        seeds.append(0x1234_5678_9ABC_DEF0)
        ctrs.append(pos | hk << 32)
        subs.append(b | ep << 32)
    inp = "".join(f"{s} {u} {c}\n" for s, u, c in zip(seeds, subs, ctrs))
    p = subprocess.run([str(exe)], input=inp, text=True, capture_output=True, timeout=120)
    assert p.returncode == 0, p.stderr
    lines = p.stdout.split("\n")
    for i, (s, u, c) in enumerate(zip(seeds, subs, ctrs)):
        got = [int(x, 16) for x in lines[i].split()]
        ctr = [c & 0xFFFFFFFF, c >> 32, u & 0xFFFFFFFF, u >> 32]
        key = [s & 0xFFFFFFFF, s >> 32]
        assert list(orc.philox4x32_10(ctr, key)) == got, (s, u, c)
