#!/usr/bin/env python3
"""Benchmark of the compressed-KV decode path on GB300.

Workload (N=1): the heavy-load LLaMA3-70B-shaped layer -- GQA 64 query / 8 KV heads,
head_dim 128, batch 512, KV length 2048, fp16 N(0,1) from a seed.  One timed step is
one decode step of every method on that batch, all through the C ABI:
  FP16      append the new token, attend over the full cache
  H2O-512   append, attend with the score update fused (logits on chip), evict to 64 + 448
  KIVI-4    append (quantising a group when the residual fills), attend
  Stream-512 append, attend, evict to 64 sinks + 448 recent
value = tokens produced per second by the whole step (4 methods x batch per step).
The H2O prefill score pass over the 2048-token prompt and the random eviction of the
reasoning-trace workload are timed in the same run and reported under "rows".

--impl reference times the fp64 CPU oracle on the host's cores on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "compressed-KV decode attn tokens/s and achieved HBM GB/s (% of ~8 TB/s), 1 GB300"
UNIT = "tokens/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _tensor_peak():
    """(dense 16-bit tensor TFLOP/s for a kernel timed alone, max SM MHz): measured, else the
    fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), float(d.get("sm_max_mhz", 2070.0))
    return 1900.0, 2070.0


def _tensor_peak_sustained():
    """Dense 16-bit tensor TFLOP/s held for seconds under the power cap: measured, else the
    fallback figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))
    return 1700.0


# ------------------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 10:   # sampler is up before timing
                time.sleep(0.01)
            self.n_before = len(self.lines)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[getattr(self, "n_before", 0):]:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------ GPU arm

class L2Flush:
    """Evicts the workload from the 129 MB L2 between timed repetitions: a write of a buffer
    larger than L2, then a read of another one, so that the timed kernel starts with L2 full
    of clean lines of unrelated data.  (A write alone leaves L2 full of dirty lines, and the
    next kernel pays for their write-back: on the 8-sequence LLaMA-7B-shaped attention that
    added ~15 us to a 45 us read.)"""

    def __init__(self, dev, nbytes: int = 512 << 20):
        import torch
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.add_(1)
        self.r.sum()


def in_graph_ms(stream, fn, flush, reset=None, R=10):
    """Milliseconds one call of fn adds to a CUDA graph of R repetitions of [reset, L2 flush,
    fn], against the same graph without fn (median of three replays each): the kernel's cost
    as it runs inside a captured decode step, without the host launch latency that an
    isolated event pair around one launch also measures (~4-5 us on this system)."""
    import torch
    graphs = []
    for with_fn in (True, False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(R):
                if reset is not None:
                    reset()
                flush()
                if with_fn:
                    fn()
        graphs.append(g)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = ([], [])
    with torch.cuda.stream(stream):
        for _ in range(3):
            for g, t in zip(graphs, ts):
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
                t.append(e0.elapsed_time(e1))
    del graphs
    return (statistics.median(ts[0]) - statistics.median(ts[1])) / R


def slot_bytes(n_slots, B, Hkv, Hq, D):
    """Algorithmic bytes of one slot-cache attention launch: K and V of the attended slots,
    the queries and the outputs."""
    return B * Hkv * n_slots * D * 2 * 2 + 2 * B * Hq * D * 2


# DRAM bytes (read + write) per (sequence, KV head) unit and cached token that ncu measured
# for k_attend_slots on the FP16 cache (64-sequence case of the heavy-load workload:
# dram__bytes_read.sum + dram__bytes_write.sum = 538.0 + 4.0 MB over 64 x 8 units x 2048 tokens).
SLOT_ATTEND_DRAM_BYTES_PER_UNIT_TOKEN = 542.0e6 / (64 * 8 * 2048)


def kivi_bytes(T, R, B, Hkv, Hq, D, bits):
    G = 32
    n_q = G * (max(0, T - R) // G)
    block = G * D * bits // 8 + 4 * D
    ring = (R + G) * D * 2 * 2
    return B * Hkv * ((n_q // G) * 2 * block + ring) + 2 * B * Hq * D * 2


def _parse_cpulist(txt: str) -> set:
    cpus = set()
    for part in txt.strip().split(","):
        if not part:
            continue
        a, _, b = part.partition("-")
        cpus.update(range(int(a), int(b or a) + 1))
    return cpus


def bind_gpu_local_cpus(dev) -> dict:
    """Run on the CPU cores next to the GPU (those of them this process may use): pinned host
    buffers land in the memory of the node whose core first touches them, and host<->device
    copies from a far node cross the CPU interconnect.  Best effort; reports what it found."""
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        bdf = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        base = os.path.join("/sys/bus/pci/devices", bdf)
        with open(os.path.join(base, "local_cpulist")) as f:
            local = _parse_cpulist(f.read())
        with open(os.path.join(base, "numa_node")) as f:
            node = int(f.read())
        allowed = os.sched_getaffinity(0)
        use = local & allowed
        if use and use != allowed:
            os.sched_setaffinity(0, use)
        return {"gpu_numa_node": node, "gpu_local_cpus": len(local), "allowed_cpus": len(allowed),
                "bound_to": len(use) if use else len(allowed)}
    except (OSError, ValueError, AttributeError) as e:
        return {"unknown": str(e)[:100]}


def run_gpu(args, rank, world):
    import torch
    import kv_cache_compression_split_gb300 as kvc
    from kv_cache_compression_split_gb300 import build as kbuild
    from kv_cache_compression_split_gb300 import workloads as W

    kbuild.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    host_binding = bind_gpu_local_cpus(dev)
    stream = torch.cuda.Stream(dev)
    w = W.HEAVY
    B, Hq, Hkv, D, T0 = w.B, w.Hq, w.Hkv, w.D, w.T
    # warm-up steps, the graph-timed steps, then as many again with per-call events
    S_total = args.warmup + 3 * args.steps
    g = Hq // Hkv
    n_heavy, n_recent, n_sink = w.n_heavy, w.n_recent, w.n_sink
    rows = {}

    with torch.cuda.stream(stream):
        # ---------------- set-up (untimed): prompt caches of 2047 tokens, then each
        # timed step appends token number 2048, 2049, ...
        K, V = W.kv_tensors(w, T=T0 - 1, device=dev, seed_offset=rank)
        Cfp = T0 + S_total + 8
        fp = kvc.SlotCache.empty(B, Hkv, Cfp, D, device=dev)
        kvc.kvc_append(fp, K, V, stream=stream)

        # H2O: prefill score pass over the prompt (timed as its own row), evict to 512
        Qp = W.q_tensor(w, device=dev, L=T0 - 1, seed_offset=rank)
        scores_full = torch.zeros(B, Hkv, Cfp, dtype=torch.float32, device=dev)
        ws_pre = torch.empty(kvc.kvc_h2o_workspace_size(B, Hq, T0 - 1) // 4, dtype=torch.float32,
                             device=dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        kvc.kvc_h2o_accumulate_prefill(Qp, fp.K, scores_full, ws_pre, T0 - 1, stream=stream)
        pre_ms = []
        pre_clk = ClockSampler(dev.index)   # the pass runs long enough to meet the power cap
        pre_clk.start()
        for _ in range(5):
            ev0.record(stream)
            kvc.kvc_h2o_accumulate_prefill(Qp, fp.K, scores_full, ws_pre, T0 - 1, stream=stream)
            ev1.record(stream)
            ev1.synchronize()
            pre_ms.append(ev0.elapsed_time(ev1))
        pre_clocks = pre_clk.stop()
        L = T0 - 1
        flops = 2 * 2 * B * Hq * (L * (L + 1) // 2) * D
        # two bounds: the tensor cores (QK^T twice) and the SFU (one exp2 per causal score in
        # each pass), which issues 32 exp2 per clock per SM on this GPU (a throughput loop of
        # independent ex2.approx chains sustains ~30 at 2.07 GHz)
        exps = 2 * B * Hq * (L * (L + 1) // 2)
        tensor_tflops, sm_mhz = _tensor_peak()
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        t_tensor = flops / (tensor_tflops * 1e12) * 1e3
        t_sfu = exps / (n_sm * 32 * sm_mhz * 1e6) * 1e3
        rows["h2o_prefill_score_pass"] = {
            "ms": min(pre_ms), "tflops": flops / (min(pre_ms) * 1e-3) / 1e12,
            "frac_of_tensor_peak": t_tensor / min(pre_ms),
            "frac_of_sustained_tensor_peak":
                flops / (min(pre_ms) * 1e-3) / 1e12 / _tensor_peak_sustained(),
            "clocks": pre_clocks, "exp2": exps,
            "sfu_bound_ms": t_sfu, "tensor_bound_ms": t_tensor,
            "frac_of_bound": max(t_sfu, t_tensor) / min(pre_ms),
            "shape": f"Qp[{B},{Hq},{L},{D}] x Kp[{B},{Hkv},{L},{D}], causal, two passes"}
        # the same scores with the rows' normalisers supplied (a causal flash-attention
        # forward over the prompt returns them), so only the column-sum pass runs; the
        # normalisers come from the two-pass call's workspace (-lse in log2 units)
        Lpad = (L + 127) // 128 * 128
        lse_rows = (ws_pre[:B * Hq * Lpad].view(B, Hq, Lpad)[:, :, :L] * (-math.log(2.0)))
        lse_rows = lse_rows.contiguous()
        kvc.kvc_h2o_accumulate_prefill(Qp, fp.K, scores_full, ws_pre, L, lse=lse_rows,
                                       stream=stream)
        one_ms = []
        for _ in range(5):
            ev0.record(stream)
            kvc.kvc_h2o_accumulate_prefill(Qp, fp.K, scores_full, ws_pre, L, lse=lse_rows,
                                           stream=stream)
            ev1.record(stream)
            ev1.synchronize()
            one_ms.append(ev0.elapsed_time(ev1))
        rows["h2o_prefill_score_pass_given_lse"] = {
            "ms": min(one_ms), "tflops": flops / 2 / (min(one_ms) * 1e-3) / 1e12,
            "frac_of_tensor_peak": t_tensor / 2 / min(one_ms),
            "frac_of_sustained_tensor_peak":
                flops / 2 / (min(one_ms) * 1e-3) / 1e12 / _tensor_peak_sustained(),
            "shape": f"Qp[{B},{Hq},{L},{D}] x Kp[{B},{Hkv},{L},{D}], causal, the column-sum "
                     f"pass only (row normalisers supplied)"}
        del Qp, ws_pre, lse_rows
        Ch = 520
        tmp = kvc.SlotCache(K=fp.K.clone(), V=fp.V.clone(), pos=fp.pos.clone(), n=fp.n.clone(),
                            seqlen=fp.seqlen.clone())
        kvc.kvc_h2o_evict(tmp, scores_full, n_heavy, n_recent, stream=stream)
        h2o = kvc.SlotCache.empty(B, Hkv, Ch, D, device=dev)
        h2o.K[:, :, :512] = tmp.K[:, :, :512]
        h2o.V[:, :, :512] = tmp.V[:, :, :512]
        h2o.pos[:, :, :512] = tmp.pos[:, :, :512]
        h2o.n.copy_(tmp.n)
        h2o.seqlen.copy_(tmp.seqlen)
        h2o_scores = torch.zeros(B, Hkv, Ch, dtype=torch.float32, device=dev)
        h2o_scores[:, :, :512] = scores_full[:, :, :512]
        del scores_full
        # StreamingLLM: prefill gather to 64 sinks + 448 recent
        tmp.K.copy_(fp.K)
        tmp.V.copy_(fp.V)
        tmp.pos.copy_(fp.pos)
        tmp.n.copy_(fp.n)
        tmp.seqlen.copy_(fp.seqlen)
        kvc.kvc_stream_evict(tmp, n_sink, n_recent, stream=stream)
        st = kvc.SlotCache.empty(B, Hkv, Ch, D, device=dev)
        st.K[:, :, :512] = tmp.K[:, :, :512]
        st.V[:, :, :512] = tmp.V[:, :, :512]
        st.pos[:, :, :512] = tmp.pos[:, :, :512]
        st.n.copy_(tmp.n)
        st.seqlen.copy_(tmp.seqlen)
        del tmp
        # KIVI-4: the prompt through the packer
        Cq = 32 * ((T0 + S_total + KIVI_AMORT_STEPS) // 32 + 1)
        kv4 = kvc.QuantCache.empty(B, Hkv, Cq, D, 4, w.kivi_R, device=dev)
        kvc.kvc_append_quant(kv4, K, V, stream=stream)
        # GEAR-4: the same prompt through the GEAR packer (its own rows, timed after the step)
        gear4 = kvc.QuantCache.empty(B, Hkv, Cq, D, 4, w.kivi_R, device=dev, gear=True)
        rows.update(pack_rows(kvc, dev, stream, kv4, gear4, K, V))
        # KIVI-4's decode steps start on a group flush: the prompt is cut so that the token of
        # the first timed step completes a group, so a window of K steps holds ceil(K / 32)
        # flushes (one every 32 tokens, R1-R5) rather than possibly none
        kv_shift = (T0 + args.warmup - w.kivi_R) % 32
        Lk = T0 - 1 - kv_shift
        kv4.len.zero_()
        kvc.kvc_append_quant(kv4, K[:, :, :Lk].contiguous(), V[:, :, :Lk].contiguous(),
                             stream=stream)
        del K, V

        # per-step inputs, resident in HBM (distinct for every step and method)
        gq = W.generator(w.seed + 900 + rank, dev)
        qs = torch.randn(S_total, 4, B, Hq, D, generator=gq, device=dev).half()
        kn = torch.randn(S_total, 4, B, Hkv, 1, D, generator=gq, device=dev).half()
        vn = torch.randn(S_total, 4, B, Hkv, 1, D, generator=gq, device=dev).half()
        outs = torch.empty(4, B, Hq, D, dtype=torch.float16, device=dev)
        outs_base = outs
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)

        def ws_for(cache):
            nb = kvc.kvc_workspace_size(cache, qs[0, 0])
            return torch.empty(max(nb // 4, 1), dtype=torch.float32, device=dev), nb

        ws_fp, nb_fp = ws_for(fp)
        ws_h2o, nb_h2o = ws_for(h2o)
        ws_st, nb_st = ws_for(st)
        ws_kv, nb_kv = ws_for(kv4)
        # kernels per step: the FP16 append 1 + attention 1 (+1 combine with several splits);
        # the H2O and StreamingLLM decode steps 1 each (append, attention, score update and
        # eviction in one launch); the KIVI append 2 (pack + length) + attention 1 (+1)
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        h2o_launches = 1 if B * Hkv <= 4 * n_sm else 3   # kvc_h2o_decode_step's own choice
        launches_per_step = (1 + 1 + (nb_fp > 0)) + h2o_launches + (2 + 1 + (nb_kv > 0)) + 1
        torch.cuda.synchronize(dev)

    names = ["fp16_append", "fp16_attend", "h2o_step", "kivi4_append", "kivi4_attend",
             "stream_step"]

    def step(i, ev=None, outs_override=None):
        """One decode step of all four methods on the launch stream; ev: per-call events."""
        outs = outs_base if outs_override is None else outs_override

        def mark(k):
            if ev is not None:
                ev[k].record(stream)
        mark(0)
        kvc.kvc_append(fp, kn[i, 0], vn[i, 0], stream=stream); mark(1)
        kvc.kvc_decode_attend(fp, qs[i, 0], outs[0], workspace=ws_fp, stream=stream); mark(2)
        # H2O: append + attention + score update (logits on chip) + eviction in one call (one
        # launch, or three for batches of more than four units per SM)
        kvc.kvc_h2o_decode_step(h2o, h2o_scores, qs[i, 1], kn[i, 1], vn[i, 1], outs[1], lse,
                                n_heavy, n_recent, stream=stream); mark(3)
        kvc.kvc_append_quant(kv4, kn[i, 2], vn[i, 2], stream=stream); mark(4)
        kvc.kvc_decode_attend(kv4, qs[i, 2], outs[2], workspace=ws_kv, stream=stream); mark(5)
        # StreamingLLM: attention without the token that left; its slot takes the new one
        kvc.kvc_stream_decode_step(st, qs[i, 3], kn[i, 3], vn[i, 3], outs[3], None, n_sink,
                                   n_recent, stream=stream); mark(6)

    branches = [torch.cuda.Stream(dev) for _ in range(4)]

    def step_par(i, outs_override=None):
        """One decode step of the four methods, each on its own stream, forked from and joined
        back into the launch stream (the methods share no data; each method's launches stay in
        order on its stream)."""
        outs = outs_base if outs_override is None else outs_override
        fork = torch.cuda.Event()
        fork.record(stream)
        for bs in branches:
            bs.wait_event(fork)
        s0, s1, s2, s3 = branches
        kvc.kvc_append(fp, kn[i, 0], vn[i, 0], stream=s0)
        kvc.kvc_decode_attend(fp, qs[i, 0], outs[0], workspace=ws_fp, stream=s0)
        kvc.kvc_h2o_decode_step(h2o, h2o_scores, qs[i, 1], kn[i, 1], vn[i, 1], outs[1], lse,
                                n_heavy, n_recent, stream=s1)
        kvc.kvc_append_quant(kv4, kn[i, 2], vn[i, 2], stream=s2)
        kvc.kvc_decode_attend(kv4, qs[i, 2], outs[2], workspace=ws_kv, stream=s2)
        kvc.kvc_stream_decode_step(st, qs[i, 3], kn[i, 3], vn[i, 3], outs[3], None, n_sink,
                                   n_recent, stream=s3)
        for bs in branches:
            join = torch.cuda.Event()
            join.record(bs)
            stream.wait_event(join)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---------------- device-resident timing
    # The K timed steps are captured once into a CUDA graph (every launch of all four
    # methods; each step forks the methods onto four streams and joins them) and the graph
    # is launched once inside the timed region, so the step time carries no host launch
    # gaps.  K more steps captured with the methods one after another on the launch stream
    # give the serial step time, and K fresh steps launched eagerly with an event between
    # calls give the per-kernel breakdown.
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step_par(i)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for k in range(args.steps):
                step_par(args.warmup + k)
        graph_ser = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ser, stream=stream):
            for k in range(args.steps):
                step(args.warmup + args.steps + k)
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        clk = ClockSampler(dev.index)
        clk.start()
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        graph.replay()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        clocks = clk.stop()
        barrier()
        s_start, s_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_start.record(stream)
        graph_ser.replay()
        s_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
               for _ in range(args.steps)]
        for k in range(args.steps):
            step(args.warmup + 2 * args.steps + k, ev=evs[k])
        torch.cuda.synchronize(dev)
        del graph, graph_ser
    total_ms = t_start.elapsed_time(t_end)
    serial_ms = s_start.elapsed_time(s_end)
    per_call = {nm: [] for nm in names}
    for k in range(args.steps):
        for j, nm in enumerate(names):
            per_call[nm].append(evs[k][j].elapsed_time(evs[k][j + 1]))
    status = kvc.kvc_read_device_status(stream)

    # algorithmic bytes per step of each attention launch (sizes of the timed steps)
    hbm_peak, peak_kind = _peaks()
    steps_T = [T0 + args.warmup + 2 * args.steps + k for k in range(args.steps)]   # FP16 tokens attended
    b_fp = [slot_bytes(t, B, Hkv, Hq, D) for t in steps_T]
    b_h2o = slot_bytes(513, B, Hkv, Hq, D)
    b_st = slot_bytes(513, B, Hkv, Hq, D)
    kv_T = [t - kv_shift for t in steps_T]   # KIVI-4 tokens attended (its prompt is shorter)
    b_kv = [kivi_bytes(t, w.kivi_R, B, Hkv, Hq, D, 4) for t in kv_T]
    ms = lambda nm: sum(per_call[nm])
    # the H2O step also reads and writes the 513 scores of every unit and writes one row
    b_h2o_step = b_h2o + B * Hkv * 513 * 4 * 2 + B * Hkv * D * 2 * 2
    b_st_step = b_st + B * Hkv * D * 2 * 2
    slot_bytes_total = sum(b_fp) + b_h2o_step * args.steps + b_st_step * args.steps
    slot_ms = ms("fp16_attend") + ms("h2o_step") + ms("stream_step")
    kernels = {
        "attend_slots(fp16+h2o+stream)": {"bytes_per_step": slot_bytes_total / args.steps,
                                          "ms_per_step": slot_ms / args.steps},
        "attend_fp16": {"bytes_per_step": sum(b_fp) / args.steps,
                        "ms_per_step": ms("fp16_attend") / args.steps},
        "attend_h2o512": {"bytes_per_step": b_h2o_step, "ms_per_step": ms("h2o_step") / args.steps,
                          "launch": "kvc_h2o_decode_step: append + attention + score update + "
                                    "eviction (three launches at this batch)"},
        "attend_stream512": {"bytes_per_step": b_st_step, "ms_per_step": ms("stream_step") / args.steps,
                             "launch": "kvc_stream_decode_step: append + attention"},
        "attend_kivi4": {"bytes_per_step": sum(b_kv) / args.steps,
                         "ms_per_step": ms("kivi4_attend") / args.steps},
    }
    for kd in kernels.values():
        kd["gbs"] = kd["bytes_per_step"] / (kd["ms_per_step"] * 1e-3) / 1e9
        kd["frac_of_hbm"] = kd["gbs"] / hbm_peak

    def spread(nm):
        v = sorted(per_call[nm])
        q = lambda f: v[min(len(v) - 1, int(f * (len(v) - 1) + 0.5))]
        return {"ms_median": statistics.median(v), "ms_p10": q(0.1), "ms_p90": q(0.9)}
    for key, nm in (("attend_fp16", "fp16_attend"), ("attend_h2o512", "h2o_step"),
                    ("attend_stream512", "stream_step"), ("attend_kivi4", "kivi4_attend")):
        kernels[key].update(spread(nm))
    methods = {
        "fp16": ms("fp16_append") + ms("fp16_attend"),
        "h2o512": ms("h2o_step"),
        "kivi4": ms("kivi4_append") + ms("kivi4_attend"),
        "stream512": ms("stream_step"),
    }
    methods = {k: {"ms_per_step": v / args.steps, "tokens_per_s": B / (v / args.steps * 1e-3)}
               for k, v in methods.items()}
    for k, v in methods.items():
        v["speedup_vs_fp16"] = methods["fp16"]["ms_per_step"] / v["ms_per_step"]
    calls = {nm: sum(v) / len(v) for nm, v in per_call.items()}

    # ---------------- end to end: host buffers, copies inside the timed region.
    # Every step uploads its own queries and new K/V from pinned host memory and reads its
    # four outputs back; uploads of step k+1 run on a copy stream while step k computes, and
    # outputs alternate between two device buffers.  The n_e2e steps, copies included, are
    # captured in one CUDA graph (replayed once to warm up, the growing caches rewound, then
    # replayed once inside the timed region), so no host launch gaps enter the number.
    n_e2e = max(3, min(args.steps, 32))   # the first upload and the last read-back are not overlapped
    base = S_total - n_e2e
    host_in = [{"q": torch.empty(4, B, Hq, D, dtype=torch.float16).pin_memory(),
                "k": torch.empty(4, B, Hkv, 1, D, dtype=torch.float16).pin_memory(),
                "v": torch.empty(4, B, Hkv, 1, D, dtype=torch.float16).pin_memory()}
               for _ in range(n_e2e)]
    host_out = [torch.empty(4, B, Hq, D, dtype=torch.float16).pin_memory() for _ in range(n_e2e)]
    for k in range(n_e2e):
        host_in[k]["q"].copy_(qs[base + k].cpu())
        host_in[k]["k"].copy_(kn[base + k].cpu())
        host_in[k]["v"].copy_(vn[base + k].cpu())
    outs2 = [outs, torch.empty_like(outs)]
    # uploads and read-backs on two streams, so that they run on different copy engines at
    # the same time (queued on one stream, the two together outlast a step)
    copy_stream = torch.cuda.Stream(dev)
    copy_out_stream = torch.cuda.Stream(dev)

    def rewind():
        # the FP16 and KIVI caches grow by one token per step: step indices base .. S_total
        # are replayed, so their lengths go back by n_e2e first
        with torch.cuda.stream(stream):
            fp.n.sub_(n_e2e)
            fp.seqlen.sub_(n_e2e)
            kv4.len.sub_(n_e2e)

    rewind()
    torch.cuda.synchronize(dev)
    ev_in = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_done = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_free = [torch.cuda.Event() for _ in range(n_e2e)]

    def upload(k):
        with torch.cuda.stream(copy_stream):
            qs[base + k].copy_(host_in[k]["q"], non_blocking=True)
            kn[base + k].copy_(host_in[k]["k"], non_blocking=True)
            vn[base + k].copy_(host_in[k]["v"], non_blocking=True)
            ev_in[k].record(copy_stream)

    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_e2e, stream=stream):
            fork = torch.cuda.Event()
            fork.record(stream)
            copy_stream.wait_event(fork)
            upload(0)
            for k in range(n_e2e):
                if k + 1 < n_e2e:
                    upload(k + 1)
                o_buf = outs2[k % 2]
                stream.wait_event(ev_in[k])
                if k >= 2:
                    stream.wait_event(ev_free[k - 2])   # that output buffer has been read back
                step_par(base + k, outs_override=o_buf)
                ev_done[k].record(stream)
                with torch.cuda.stream(copy_out_stream):
                    copy_out_stream.wait_event(ev_done[k])
                    host_out[k].copy_(o_buf, non_blocking=True)
                    ev_free[k].record(copy_out_stream)
            join, join_out = torch.cuda.Event(), torch.cuda.Event()
            join.record(copy_stream)
            join_out.record(copy_out_stream)
            stream.wait_event(join)
            stream.wait_event(join_out)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):   # replay() launches on the current stream
        g_e2e.replay()
    torch.cuda.synchronize(dev)
    # three timed replays, the caches rewound before each; the median is reported (the
    # host-memory side of the copies shares the machine with other jobs, and a single
    # replay once in a few runs came out 1.5-2x slower)
    e2e_runs = []
    for _ in range(3):
        rewind()
        torch.cuda.synchronize(dev)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g_e2e.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_runs.append(e0.elapsed_time(e1) / n_e2e)
    del g_e2e
    e2e_ms = statistics.median(e2e_runs)
    h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
    d2h = host_out[0].numel() * host_out[0].element_size()

    # ---------------- H2O variants and random eviction rows, timed in the same run
    rows.update(h2o_variant_rows(kvc, dev, stream, h2o, h2o_scores, qs[:, 1], kn[:, 1], vn[:, 1],
                                 n_heavy, n_recent))
    rows.update(random_rows(kvc, W, dev, stream, hbm_peak))
    rows.update(paged_rows(kvc, dev, stream, fp, kv4, qs[0, 0], T0))
    rows.update(gear_rows(kvc, dev, stream, gear4, qs[:, 2], kn[:, 2], vn[:, 2], hbm_peak))
    del gear4
    rows.update(kivi_amortized_rows(kvc, dev, stream, kv4, qs[:, 2], kn[:, 2], vn[:, 2], hbm_peak))
    rows.update(config_rows(kvc, W, dev, stream, hbm_peak))

    ms_per_step = total_ms / args.steps
    eager_ms = evs[0][0].elapsed_time(evs[-1][len(names)]) / args.steps
    # the whole timed step against the copy bandwidth: the four attention launches' bytes at
    # the timed steps' own cache lengths
    graph_T = [T0 + args.warmup + k for k in range(args.steps)]
    step_bytes = (sum(slot_bytes(t, B, Hkv, Hq, D) +
                      kivi_bytes(t - kv_shift, w.kivi_R, B, Hkv, Hq, D, 4)
                      for t in graph_T) / args.steps + b_h2o_step + b_st_step)
    step_roofline = {"bytes_per_step": step_bytes,
                     "gbs": step_bytes / (ms_per_step * 1e-3) / 1e9,
                     "frac_of_hbm": step_bytes / (ms_per_step * 1e-3) / 1e9 / hbm_peak}
    t_avg = sum(steps_T) / len(steps_T)
    fp16_traffic = SLOT_ATTEND_DRAM_BYTES_PER_UNIT_TOKEN * B * Hkv * t_avg
    res = {
        "fp16_traffic": fp16_traffic,
        "ms_per_step": ms_per_step, "serial_ms_per_step": serial_ms / args.steps,
        "step_roofline": step_roofline,
        "eager_ms_per_step": eager_ms, "e2e_ms_per_step": e2e_ms, "e2e_runs_ms": e2e_runs,
        "calls_ms": calls,
        "kernels": kernels, "methods": methods, "rows": rows, "clocks": clocks,
        "device_status": status, "tokens_per_step": 4 * B,
        "launches_per_step": launches_per_step, "h2d": h2d, "d2h": d2h,
        "host_binding": host_binding,
        "hbm_peak": hbm_peak, "peak_kind": peak_kind,
        "splits": {"fp16": nb_fp, "h2o": nb_h2o, "stream": nb_st, "kivi": nb_kv},
        "kivi_window": {"first_timed_T": graph_T[0] - kv_shift,
                        "flushes_in_timed_window":
                            sum(1 for t in graph_T if (t - kv_shift - w.kivi_R) % 32 == 0)},
    }
    return res


def h2o_variant_rows(kvc, dev, stream, src, src_scores, qs, kn, vn, n_heavy, n_recent):
    """The two H2O variants of "Practical Online KV Cache Compaction for LLM Agents" on the
    heavy-load H2O-512 state: the decayed activity score (decay 0.99, §4.1) with an eviction every
    step, and batched eviction (trigger at 110% of the 512 budget, §5.2) with plain scores.  Each
    step is append + attention with the fused score update (+ eviction); two full trigger cycles
    (2 x 51 steps) are timed, so the batched row's cost is amortised over its compactions."""
    import torch
    B, Hkv, _, D = src.K.shape
    Hq = qs.shape[2]
    budget = n_heavy + n_recent
    trigger = (11 * budget + 9) // 10           # first count above 110%: 564 for 512
    steps = 2 * (trigger - budget)
    C = trigger + 8
    out = {}
    with torch.cuda.stream(stream):
        o = torch.empty(B, Hq, D, dtype=torch.float16, device=dev)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
        for name, decay, trig in (("h2o512_decay", 0.99, None), ("h2o512_batched", 0.0, trigger)):
            c = kvc.SlotCache.empty(B, Hkv, C, D, device=dev)
            c.K[:, :, :budget] = src.K[:, :, :budget]
            c.V[:, :, :budget] = src.V[:, :, :budget]
            c.pos[:, :, :budget] = src.pos[:, :, :budget]
            c.n.copy_(src.n)
            c.seqlen.copy_(src.seqlen)
            sc = torch.zeros(B, Hkv, C, dtype=torch.float32, device=dev)
            sc[:, :, :budget] = src_scores[:, :, :budget]
            ws = torch.empty(max(kvc.kvc_workspace_size(c, qs[0], 1) // 4, 1), dtype=torch.float32,
                             device=dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record(stream)
            for i in range(steps):
                k = i % qs.shape[0]
                if trig is None:   # decayed scores, eviction every step: the one-launch step
                    kvc.kvc_h2o_decode_step(c, sc, qs[k], kn[k], vn[k], o, lse, n_heavy, n_recent,
                                            decay, stream=stream)
                    continue
                kvc.kvc_append(c, kn[k], vn[k], stream=stream)
                kvc.kvc_decode_attend(c, qs[k], o, lse=lse, workspace=ws, num_splits=1,
                                      h2o_scores=sc, h2o_decay=decay, stream=stream)
                kvc.kvc_h2o_evict_when(c, sc, n_heavy, n_recent, trig, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / steps
            out[name] = {"ms_per_step": ms, "tokens_per_s": B / (ms * 1e-3), "steps": steps,
                         "shape": f"B={B} GQA {Hq}/{Hkv} D={D}, budget {budget}" +
                                  (f", decay {decay}, evict every step (kvc_h2o_decode_step)"
                                   if trig is None else
                                   f", evict when n >= {trig} (slots attended {budget + 1}.."
                                   f"{trig})")}
            del c, sc, ws
    return out


KIVI_AMORT_STEPS = 64   # two flushes of a 32-token group


def kivi_amortized_rows(kvc, dev, stream, kv4, qs, kn, vn, hbm_peak):
    """KIVI-4 decode with its periodic group flush amortised: KIVI_AMORT_STEPS consecutive
    decode steps (append + attention; every 32nd append quantises and packs the group that
    leaves the fp16 residual) captured in one CUDA graph and timed as a whole, so the per-step
    figure carries exactly two flushes per 64 steps."""
    import torch
    B, Hkv, D, R = kv4.B, kv4.Hkv, kv4.D, kv4.R
    Hq = qs.shape[2]
    S = KIVI_AMORT_STEPS
    out = {}
    with torch.cuda.stream(stream):
        o = torch.empty(B, Hq, D, dtype=torch.float16, device=dev)
        ws = torch.empty(max(kvc.kvc_workspace_size(kv4, qs[0]) // 4, 1), dtype=torch.float32,
                         device=dev)
        T_start = int(kv4.len[0].item())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(S):
                k = i % qs.shape[0]
                kvc.kvc_append_quant(kv4, kn[k], vn[k], stream=stream)
                kvc.kvc_decode_attend(kv4, qs[k], o, workspace=ws, stream=stream)
        torch.cuda.synchronize(dev)
        kv4.len.fill_(T_start)   # capture ran nothing; the replay appends S tokens
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        del g
        ms = e0.elapsed_time(e1) / S
        flushes = sum(1 for t in range(T_start + 1, T_start + S + 1) if (t - R) % 32 == 0)
        nbytes = sum(kivi_bytes(t, R, B, Hkv, Hq, D, 4) for t in range(T_start + 1, T_start + S + 1)) / S
    out["kivi4_decode_amortized"] = {
        "ms_per_step": ms, "tokens_per_s": B / (ms * 1e-3), "steps": S, "flushes": flushes,
        "attend_bytes_per_step": nbytes,
        "step_gbs": nbytes / (ms * 1e-3) / 1e9, "step_frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm_peak,
        "shape": f"B={B} GQA {Hq}/{Hkv} D={D}, T={T_start + 1}..{T_start + S}, R={R}: "
                 f"append (+ group flush every 32 tokens) + attention, one CUDA graph"}
    return out


def pack_rows(kvc, dev, stream, kv4, gear4, K, V):
    """Bulk pack of the heavy-load prompt (B x Hkv units of 2047 tokens): KIVI-4 blocks alone,
    and KIVI-4 blocks plus the GEAR side blocks (2% sparse + rank-2 per group and side).  Each
    cache is reset and repacked; the second of two packs is timed."""
    import torch
    out = {}
    with torch.cuda.stream(stream):
        for name, c in (("kivi4_pack_prompt", kv4), ("gear4_pack_prompt", gear4)):
            times = []
            for _ in range(2):
                c.len.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                kvc.kvc_append_quant(c, K, V, stream=stream)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                times.append(e0.elapsed_time(e1))
            B, Hkv, T, D = K.shape
            out[name] = {"ms": times[-1], "tokens": B * Hkv * T,
                         "groups_per_s": B * Hkv * (T - kv4.R) // 32 / (times[-1] * 1e-3),
                         "shape": f"[{B},{Hkv},{T},{D}] fp16 -> 4-bit groups of 32 + ring"}
    return out


def gear_rows(kvc, dev, stream, gear4, qs, kn, vn, hbm_peak):
    """GEAR-4 decode on the heavy-load workload: each step appends one token (the 32nd of a
    group flushes it through the GEAR packer) and attends over the quantised groups with
    their sparse and rank-2 corrections plus the fp16 ring.  Attention bytes: KIVI-4 blocks,
    the two side blocks of every group, the ring, queries and outputs."""
    import torch
    B, Hkv, D, R = gear4.B, gear4.Hkv, gear4.D, gear4.R
    Hq = qs.shape[2]
    side = kvc.kvc_gear_side_bytes(D)
    steps = min(qs.shape[0], 40)
    out = {}
    with torch.cuda.stream(stream):
        o = torch.empty(B, Hq, D, dtype=torch.float16, device=dev)
        ws = torch.empty(max(kvc.kvc_workspace_size(gear4, qs[0]) // 4, 1), dtype=torch.float32,
                         device=dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        lens = []
        for i in range(steps):
            ev[i][0].record(stream)
            kvc.kvc_append_quant(gear4, kn[i], vn[i], stream=stream)
            ev[i][1].record(stream)
            kvc.kvc_decode_attend(gear4, qs[i], o, workspace=ws, stream=stream)
            ev[i][2].record(stream)
            lens.append(int(gear4.len[0].item()) if i == 0 else lens[-1] + 1)
        torch.cuda.synchronize(dev)
        att = [ev[i][1].elapsed_time(ev[i][2]) for i in range(1, steps)]
        app = [ev[i][0].elapsed_time(ev[i][1]) for i in range(1, steps)]
        nbytes = [kivi_bytes(t, R, B, Hkv, Hq, D, 4) +
                  B * Hkv * (max(0, t - R) // 32) * 2 * side for t in lens[1:]]
        ms_att = sum(att) / len(att)
        gbs = sum(nbytes) / len(nbytes) / (ms_att * 1e-3) / 1e9
        out["gear4_decode"] = {
            "ms_per_step": (sum(att) + sum(app)) / len(att), "attend_ms": ms_att,
            "append_ms": sum(app) / len(app), "tokens_per_s": B / ((sum(att) + sum(app)) /
                                                                  len(att) * 1e-3),
            "attend_gbs": gbs, "attend_frac_of_hbm": gbs / hbm_peak,
            "attend_bytes": sum(nbytes) / len(nbytes), "steps": steps - 1,
            "shape": f"B={B} GQA {Hq}/{Hkv} D={D}, T={lens[1]}..{lens[-1]}, R={R}, "
                     f"side block {side} B per group and side"}
    return out


def config_rows(kvc, W, dev, stream, hbm_peak):
    """Decode attention on the two MHA workloads (median of 5 after one warm-up, L2 flushed
    before each by a 512 MB write and a 512 MB read, as their compressed caches fit in L2):
    llama7b-b8-h32-d128-t2048 (FP16 over T+1 slots; H2O-512 from the prefill score pass and
    StreamingLLM-512 from the prompt gather, each over 513 slots in its decode step) and
    kivi-b32-h32-d128-t4096 (FP16, KIVI-4 and KIVI-2 over T tokens)."""
    import torch
    flush = L2Flush(dev)
    out = {}

    def timed(fn):
        ts = []
        for r in range(6):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if r > 0:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    with torch.cuda.stream(stream):
        # ---- llama7b-b8-h32-d128-t2048: 32 MHA heads, 2% outlier channels in K and V.
        # FP16 attends over the 2048-token prompt + the new token.  H2O-512: the prefill score
        # pass over the 2048-token causal prompt (queries ~ N(0,1)), eviction to 64 heavy + 448
        # recent, then the decode step append -> attention with the fused score update (logits
        # on chip) -> eviction 513 -> 512.  StreamingLLM-512: the prompt gathered to 64 sinks +
        # 448 recent, then the decode step kvc_stream_append -> attention.
        w = W.LLAMA7B
        B, Hq, Hkv, D, T = w.B, w.Hq, w.Hkv, w.D, w.T
        K, V = W.kv_tensors(w, T=T + 1, device=dev)
        q = W.q_tensor(w, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
        kn, vn = K[:, :, T:T + 1].contiguous(), V[:, :, T:T + 1].contiguous()
        c = kvc.SlotCache.empty(B, Hkv, T + 8, D, device=dev)
        kvc.kvc_append(c, K, V, stream=stream)
        ws = torch.empty(max(kvc.kvc_workspace_size(c, q) // 4, 1), dtype=torch.float32, device=dev)
        fn = lambda: kvc.kvc_decode_attend(c, q, o, workspace=ws, stream=stream)
        ms = timed(fn)
        mg = in_graph_ms(stream, fn, flush)
        nb = slot_bytes(T + 1, B, Hkv, Hq, D)
        out[f"{w.name}/fp16"] = {"ms": ms, "slots": T + 1, "gbs": nb / (ms * 1e-3) / 1e9,
                                 "frac_of_hbm": nb / (ms * 1e-3) / 1e9 / hbm_peak,
                                 "ms_in_graph": mg,
                                 "frac_of_hbm_in_graph": nb / (mg * 1e-3) / 1e9 / hbm_peak,
                                 "tokens_per_s": B / (ms * 1e-3)}
        del c, ws
        # the two compressed caches after the prompt (set-up, untimed)
        full = kvc.SlotCache.empty(B, Hkv, T + 8, D, device=dev)
        kvc.kvc_append(full, K[:, :, :T].contiguous(), V[:, :, :T].contiguous(), stream=stream)
        qp = W.q_tensor(w, L=T, device=dev)
        sc_full = torch.zeros(B, Hkv, T + 8, dtype=torch.float32, device=dev)
        pws = torch.empty(kvc.kvc_h2o_workspace_size(B, Hq, T) // 4, dtype=torch.float32,
                          device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush()
        e0.record(stream)
        kvc.kvc_h2o_accumulate_prefill(qp, full.K, sc_full, pws, T, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        pre_ms = e0.elapsed_time(e1)
        del qp, pws
        pos0, K0, V0, n0, sl0 = (full.pos.clone(), full.K.clone(), full.V.clone(), full.n.clone(),
                                 full.seqlen.clone())
        kvc.kvc_h2o_evict(full, sc_full, w.n_heavy, w.n_recent, stream=stream)
        Ch = 520
        h2o0 = {"K": full.K[:, :, :Ch].clone(), "V": full.V[:, :, :Ch].clone(),
                "pos": full.pos[:, :, :Ch].clone(), "n": full.n.clone(), "seqlen": full.seqlen.clone(),
                "sc": sc_full[:, :, :Ch].clone()}
        full.pos.copy_(pos0); full.K.copy_(K0); full.V.copy_(V0); full.n.copy_(n0)
        full.seqlen.copy_(sl0)
        del pos0, K0, V0, n0, sl0, sc_full
        kvc.kvc_stream_evict(full, w.n_sink, w.n_recent, stream=stream)
        st0 = {"K": full.K[:, :, :Ch].clone(), "V": full.V[:, :, :Ch].clone(),
               "pos": full.pos[:, :, :Ch].clone(), "n": full.n.clone(), "seqlen": full.seqlen.clone()}
        del full
        hc = kvc.SlotCache.empty(B, Hkv, Ch, D, device=dev)
        hsc = torch.zeros(B, Hkv, Ch, dtype=torch.float32, device=dev)
        stc = kvc.SlotCache.empty(B, Hkv, Ch, D, device=dev)
        ws_h = torch.empty(max(kvc.kvc_workspace_size(hc, q) // 4, 1), dtype=torch.float32,
                           device=dev)

        def reset_h2o():
            for k_ in ("K", "V", "pos", "n", "seqlen"):
                getattr(hc, k_).copy_(h2o0[k_])
            hsc.copy_(h2o0["sc"])

        def reset_st():
            for k_ in ("K", "V", "pos", "n", "seqlen"):
                getattr(stc, k_).copy_(st0[k_])

        def step_times(reset, launches):
            """Median over 5 repetitions (one warm-up) of each launch of the step, the cache
            reset and L2 flushed before each repetition."""
            ts = [[] for _ in launches]
            for r in range(6):
                reset()
                flush()
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)]
                evs[0].record(stream)
                for j, fn in enumerate(launches):
                    fn()
                    evs[j + 1].record(stream)
                evs[-1].synchronize()
                if r > 0:
                    for j in range(len(launches)):
                        ts[j].append(evs[j].elapsed_time(evs[j + 1]))
            return [statistics.median(t) for t in ts]

        t_app, t_att, t_ev = step_times(reset_h2o, [
            lambda: kvc.kvc_append(hc, kn, vn, stream=stream),
            lambda: kvc.kvc_decode_attend(hc, q, o, lse=lse, workspace=ws_h, h2o_scores=hsc,
                                          stream=stream),
            lambda: kvc.kvc_h2o_evict(hc, hsc, w.n_heavy, w.n_recent, stream=stream)])
        nb = slot_bytes(513, B, Hkv, Hq, D)
        h_app = lambda: kvc.kvc_append(hc, kn, vn, stream=stream)
        h_att = lambda: kvc.kvc_decode_attend(hc, q, o, lse=lse, workspace=ws_h, h2o_scores=hsc,
                                              stream=stream)
        h_ev = lambda: kvc.kvc_h2o_evict(hc, hsc, w.n_heavy, w.n_recent, stream=stream)
        g_att = in_graph_ms(stream, h_att, flush, reset=lambda: (reset_h2o(), h_app()))
        g_step = in_graph_ms(stream, lambda: (h_app(), h_att(), h_ev()), flush, reset=reset_h2o)
        h_step = lambda: kvc.kvc_h2o_decode_step(hc, hsc, q, kn, vn, o, lse, w.n_heavy, w.n_recent,
                                                 stream=stream)
        (t_fused,) = step_times(reset_h2o, [h_step])
        g_fused = in_graph_ms(stream, h_step, flush, reset=reset_h2o)
        out[f"{w.name}/h2o512"] = {
            "fused_step_ms": t_fused, "fused_step_ms_in_graph": g_fused,
            "fused_step_frac_of_hbm_in_graph": nb / (g_fused * 1e-3) / 1e9 / hbm_peak,
            "ms": t_att, "slots": 513, "gbs": nb / (t_att * 1e-3) / 1e9,
            "frac_of_hbm": nb / (t_att * 1e-3) / 1e9 / hbm_peak, "tokens_per_s": B / (t_att * 1e-3),
            "ms_in_graph": g_att, "frac_of_hbm_in_graph": nb / (g_att * 1e-3) / 1e9 / hbm_peak,
            "step_ms_in_graph": g_step,
            "step_ms": t_app + t_att + t_ev, "append_ms": t_app, "evict_ms": t_ev,
            "prefill_score_pass_ms": pre_ms,
            "cache": "prefill scores of the 2048-token causal prompt, evicted to 64 heavy + "
                     "448 recent; step: append, attention + fused score update, 513 -> 512"}
        t_app, t_att = step_times(reset_st, [
            lambda: kvc.kvc_stream_append(stc, kn, vn, w.n_sink, w.n_recent, stream=stream),
            lambda: kvc.kvc_decode_attend(stc, q, o, workspace=ws_h, stream=stream)])
        s_app = lambda: kvc.kvc_stream_append(stc, kn, vn, w.n_sink, w.n_recent, stream=stream)
        s_att = lambda: kvc.kvc_decode_attend(stc, q, o, workspace=ws_h, stream=stream)
        g_att = in_graph_ms(stream, s_att, flush, reset=lambda: (reset_st(), s_app()))
        g_step = in_graph_ms(stream, lambda: (s_app(), s_att()), flush, reset=reset_st)
        s_step = lambda: kvc.kvc_stream_decode_step(stc, q, kn, vn, o, None, w.n_sink, w.n_recent,
                                                    stream=stream)
        (t_fused,) = step_times(reset_st, [s_step])
        g_fused = in_graph_ms(stream, s_step, flush, reset=reset_st)
        out[f"{w.name}/stream512"] = {
            "fused_step_ms": t_fused, "fused_step_ms_in_graph": g_fused,
            "fused_step_frac_of_hbm_in_graph": nb / (g_fused * 1e-3) / 1e9 / hbm_peak,
            "ms": t_att, "slots": 513, "gbs": nb / (t_att * 1e-3) / 1e9,
            "frac_of_hbm": nb / (t_att * 1e-3) / 1e9 / hbm_peak, "tokens_per_s": B / (t_att * 1e-3),
            "ms_in_graph": g_att, "frac_of_hbm_in_graph": nb / (g_att * 1e-3) / 1e9 / hbm_peak,
            "step_ms_in_graph": g_step,
            "step_ms": t_app + t_att, "append_ms": t_app,
            "cache": "the prompt gathered to 64 sinks + 448 recent; step: kvc_stream_append "
                     "(the leaving token's slot), attention over 513"}
        del hc, hsc, stc, ws_h, h2o0, st0, K, V
        # ---- kivi-b32-h32-d128-t4096: offsets U(-2, 2) on Q, K, V
        w = W.KIVI_MHA
        B, Hq, Hkv, D, T = w.B, w.Hq, w.Hkv, w.D, w.T
        K, V = W.kv_tensors(w, T=T, device=dev)
        q = W.q_tensor(w, device=dev)
        o = torch.empty_like(q)
        c = kvc.SlotCache.empty(B, Hkv, T + 8, D, device=dev)
        kvc.kvc_append(c, K, V, stream=stream)
        ws = torch.empty(max(kvc.kvc_workspace_size(c, q) // 4, 1), dtype=torch.float32, device=dev)
        fn = lambda: kvc.kvc_decode_attend(c, q, o, workspace=ws, stream=stream)
        ms = timed(fn)
        mg = in_graph_ms(stream, fn, flush)
        nb = slot_bytes(T, B, Hkv, Hq, D)
        out[f"{w.name}/fp16"] = {"ms": ms, "slots": T, "gbs": nb / (ms * 1e-3) / 1e9,
                                 "frac_of_hbm": nb / (ms * 1e-3) / 1e9 / hbm_peak,
                                 "ms_in_graph": mg,
                                 "frac_of_hbm_in_graph": nb / (mg * 1e-3) / 1e9 / hbm_peak,
                                 "tokens_per_s": B / (ms * 1e-3)}
        del c, ws
        for bits in (4, 2):
            kq = kvc.QuantCache.empty(B, Hkv, T, D, bits, w.kivi_R, device=dev)
            kvc.kvc_append_quant(kq, K, V, stream=stream)
            ws = torch.empty(max(kvc.kvc_workspace_size(kq, q) // 4, 1), dtype=torch.float32,
                             device=dev)
            fn = lambda: kvc.kvc_decode_attend(kq, q, o, workspace=ws, stream=stream)
            ms = timed(fn)
            mg = in_graph_ms(stream, fn, flush)
            nb = kivi_bytes(T, w.kivi_R, B, Hkv, Hq, D, bits)
            out[f"{w.name}/kivi{bits}"] = {"ms": ms, "tokens": T, "gbs": nb / (ms * 1e-3) / 1e9,
                                           "frac_of_hbm": nb / (ms * 1e-3) / 1e9 / hbm_peak,
                                           "ms_in_graph": mg,
                                           "frac_of_hbm_in_graph":
                                               nb / (mg * 1e-3) / 1e9 / hbm_peak,
                                           "tokens_per_s": B / (ms * 1e-3)}
            del kq, ws
        del K, V, flush
    return out


def paged_rows(kvc, dev, stream, dense, kv4, q, T):
    """Decode attention on the heavy-load caches, dense and in the paged layout (pages of one
    pool handed out in a shuffled order), same data: FP16 over the first T slots, and KIVI-4
    (128-token pages of four group blocks) over the cache as the timed steps left it."""
    import torch
    B, Hkv, D = dense.B, dense.Hkv, dense.D
    Cp = 64 * ((T + 63) // 64)
    npu = Cp // 64
    num_pages = B * Hkv * npu
    out = {}
    with torch.cuda.stream(stream):
        perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(64))
        table = perm.to(torch.int32).view(B, Hkv, npu).to(dev)
        paged = kvc.SlotCache.empty_paged(B, Hkv, Cp, D, num_pages, block_table=table, device=dev)
        rows = (table.long()[..., None] * 64 + torch.arange(64, device=dev)).reshape(-1)
        src = dense.K[:, :, :Cp].reshape(-1, D)
        paged.K.view(-1, D)[rows] = src
        paged.V.view(-1, D)[rows] = dense.V[:, :, :Cp].reshape(-1, D)
        paged.n.fill_(T)
        paged.seqlen.fill_(T)
        view = kvc.SlotCache(K=dense.K, V=dense.V, pos=dense.pos, n=torch.full_like(dense.n, T),
                             seqlen=dense.seqlen)
        o = torch.empty_like(q)
        for name, c in (("fp16_attend_dense_T", view), ("fp16_attend_paged_T", paged)):
            ws = torch.empty(max(kvc.kvc_workspace_size(c, q) // 4, 1), dtype=torch.float32,
                             device=dev)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(6)]
            for e0, e1 in ev:
                e0.record(stream)
                kvc.kvc_decode_attend(c, q, o, workspace=ws, stream=stream)
                e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev[1:])
            out[name] = {"ms": ms, "slots": T,
                         "gbs": slot_bytes(T, B, Hkv, q.shape[1], D) / (ms * 1e-3) / 1e9,
                         "layout": "paged, 64-slot pages in shuffled order" if c is paged
                                   else "dense"}
        del paged
        # KIVI-4: the same blocks, reached through a shuffled page table
        B_, Hkv_, ng, bb = kv4.k_blocks.shape
        npu = ng // 4
        nump = B_ * Hkv_ * npu
        perm = torch.randperm(nump, generator=torch.Generator().manual_seed(128))
        ktab = perm.to(torch.int32).view(B_, Hkv_, npu).to(dev)
        pk = kvc.QuantCache.empty_paged(B_, Hkv_, npu * 128, kv4.D, kv4.bits, kv4.R, nump,
                                        block_table=ktab, device=dev)
        idx = (ktab.long()[..., None] * 4 + torch.arange(4, device=dev)).reshape(-1)
        pk.k_blocks.view(-1, bb)[idx] = kv4.k_blocks[:, :, :npu * 4].reshape(-1, bb)
        pk.v_blocks.view(-1, bb)[idx] = kv4.v_blocks[:, :, :npu * 4].reshape(-1, bb)
        pk.k_res.copy_(kv4.k_res)
        pk.v_res.copy_(kv4.v_res)
        pk.len.copy_(kv4.len)
        for name, c in (("kivi4_attend_dense", kv4), ("kivi4_attend_paged", pk)):
            ws = torch.empty(max(kvc.kvc_workspace_size(c, q) // 4, 1), dtype=torch.float32,
                             device=dev)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(6)]
            for e0, e1 in ev:
                e0.record(stream)
                kvc.kvc_decode_attend(c, q, o, workspace=ws, stream=stream)
                e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev[1:])
            out[name] = {"ms": ms, "tokens": int(kv4.len[0]),
                         "layout": "paged, 128-token pages in shuffled order" if c is pk
                                   else "dense"}
        del pk
    return out


def random_rows(kvc, W, dev, stream, hbm_peak):
    """Random eviction on the reasoning-trace workload, run as the trace runs: 16 sequences,
    GQA 64/8, a locked prompt of 1024 tokens, 1024 generated tokens appended per epoch, an
    eviction to keep 0.25 of the generated tokens per KV head at T = 2048, 3072, ..., 32768
    (31 evictions, epochs 0..30, positions up to 32767), and decode attention after every
    eviction.  L2 is flushed (a 512 MB write and a 512 MB read) before each eviction, so both
    launches read the cache from HBM; the bulk appends are set-up, not timed.  The row reports
    the steady state (epochs 5..30: 2389 -> 1365 slots per head) and every epoch's times."""
    import torch
    w = W.REASONING
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    P, every, T_end = w.prompt_len, w.evict_every, w.T
    n_evict = (T_end - P) // every
    out = {}
    with torch.cuda.stream(stream):
        K, V = W.kv_tensors(w, T=T_end, device=dev)
        C = 2432
        c = kvc.SlotCache.empty(B, Hkv, C, D, device=dev)
        kvc.kvc_append(c, K[:, :, :P + every].contiguous(), V[:, :, :P + every].contiguous(),
                       stream=stream)
        qs = [W.q_tensor(w, device=dev, seed_offset=e) for e in range(n_evict)]
        o = torch.empty_like(qs[0])
        flush = L2Flush(dev)
        t_ev, t_at, ev_bytes, at_bytes, n_before, n_after = [], [], [], [], [], []
        for e in range(n_evict):
            if e > 0:
                t0 = P + every * e
                kvc.kvc_append(c, K[:, :, t0:t0 + every].contiguous(),
                               V[:, :, t0:t0 + every].contiguous(), stream=stream)
            ws = torch.empty(max(kvc.kvc_workspace_size(c, qs[e]) // 4, 1), dtype=torch.float32,
                             device=dev)
            n0 = int(c.n[0, 0].item())
            pre = c.pos[:, :, :n0].clone()
            flush()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            kvc.kvc_random_evict(c, P, w.keep_ratio, W.RANDOM_EVICT_SEED, e, stream=stream)
            ev[1].record(stream)
            kvc.kvc_decode_attend(c, qs[e], o, workspace=ws, stream=stream)
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            n1 = int(c.n[0, 0].item())
            # rows the compaction moved: kept slots of [0, n1) whose position changed
            moved = int((c.pos[:, :, :n1] != pre[:, :, :n1]).sum().item())
            t_ev.append(ev[0].elapsed_time(ev[1]))
            t_at.append(ev[1].elapsed_time(ev[2]))
            # eviction: every slot's position read once, each moved row's K and V read and
            # written, its position written
            ev_bytes.append(B * Hkv * n0 * 4 + moved * (2 * 2 * D * 2 + 4))
            at_bytes.append(slot_bytes(n1, B, Hkv, Hq, D))
            n_before.append(n0)
            n_after.append(n1)
        # the last eviction again, inside a CUDA graph (its pre-eviction positions and count
        # restored before each repetition: the same keep-set and the same moved rows)
        n0_last = n_before[-1]

        def reset_last():
            c.pos[:, :, :n0_last].copy_(pre)
            c.n.fill_(n0_last)
        e = n_evict - 1
        g_ev = in_graph_ms(stream, lambda: kvc.kvc_random_evict(c, P, w.keep_ratio,
                                                                W.RANDOM_EVICT_SEED, e,
                                                                stream=stream),
                           flush, reset=reset_last)
        # the baseline graph ran last and left the pre-eviction state: evict once more
        reset_last()
        kvc.kvc_random_evict(c, P, w.keep_ratio, W.RANDOM_EVICT_SEED, e, stream=stream)
        torch.cuda.synchronize(dev)
        assert int(c.n[0, 0].item()) == n_after[-1]
        g_at = in_graph_ms(stream, lambda: kvc.kvc_decode_attend(c, qs[e], o, workspace=ws,
                                                                 stream=stream), flush)
        st = list(range(5, n_evict))
        ms_ev = statistics.median(t_ev[i] for i in st)
        ms_at = statistics.median(t_at[i] for i in st)
        gb_ev = statistics.median(ev_bytes[i] for i in st)
        gb_at = statistics.median(at_bytes[i] for i in st)
        assert kvc.kvc_read_device_status(stream) == 0
        del K, V, c, flush
    out["random_evict_reasoning"] = {
        "ms": ms_ev, "bytes": gb_ev, "gbs": gb_ev / (ms_ev * 1e-3) / 1e9,
        "frac_of_hbm": gb_ev / (ms_ev * 1e-3) / 1e9 / hbm_peak,
        "ms_in_graph": g_ev, "frac_of_hbm_in_graph": ev_bytes[-1] / (g_ev * 1e-3) / 1e9 / hbm_peak,
        "slots_before": n_before[-1], "kept_per_head": n_after[-1],
        "ms_per_epoch": [round(t, 4) for t in t_ev],
        "shape": f"B={B} Hkv={Hkv} D={D}, prompt {P} locked, evictions at T = {P + every}.."
                 f"{T_end} (epochs 0..{n_evict - 1}); steady state epochs 5..{n_evict - 1}: "
                 f"{n_before[-1]} -> {n_after[-1]} slots per head; L2 flushed before each"}
    out["random_attend_reasoning"] = {
        "ms": ms_at, "slots": n_after[-1], "bytes": gb_at,
        "gbs": gb_at / (ms_at * 1e-3) / 1e9, "frac_of_hbm": gb_at / (ms_at * 1e-3) / 1e9 / hbm_peak,
        "ms_in_graph": g_at, "frac_of_hbm_in_graph": at_bytes[-1] / (g_at * 1e-3) / 1e9 / hbm_peak,
        "tokens_per_s": B / (ms_at * 1e-3), "ms_per_epoch": [round(t, 4) for t in t_at]}
    return out


# ------------------------------------------------------------------------------------ CPU oracle

def oracle_prefill_sample(n_seq: int, threads: int) -> float:
    """Seconds the fp64 oracle takes for the H2O prefill score pass of n_seq sequences of the
    heavy-load prompt (2047 tokens, all 8 KV heads)."""
    import oracle as orc
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.HEAVY
    L = w.T - 1
    Qp = W.q_tensor(w, B=n_seq, L=L).numpy()
    Kp, _ = W.kv_tensors(w, T=L, B=n_seq)
    t0 = time.perf_counter()
    orc.h2o_prefill_scores(Qp, Kp.numpy(), L, threads=threads)
    return time.perf_counter() - t0


def oracle_sample(n_seq: int, threads: int):
    """Time the fp64 oracle on n_seq sequences (all 8 KV heads) of the heavy-load workload,
    one decode step of each method; returns (seconds, tokens produced = 4 * n_seq)."""
    import numpy as np
    import oracle as orc
    from kv_cache_compression_split_gb300 import workloads as W
    w = W.HEAVY
    Hq, Hkv, D, T = w.Hq, w.Hkv, w.D, w.T
    K, V = W.kv_tensors(w, T=T, B=n_seq)
    q = W.q_tensor(w, B=n_seq)
    K16, V16, q16 = K.numpy(), V.numpy(), q.numpy()
    t0 = time.perf_counter()
    # FP16: full attention over T tokens
    orc.decode_attend(q16, K16, V16, np.full((n_seq, Hkv), T), threads=threads)
    # StreamingLLM-512: keep-set, gather, attention over 513
    keep = orc.stream_keep(np.arange(T), T, w.n_sink, w.n_recent + 1)
    idx = np.flatnonzero(keep)
    Ks, Vs = K16[:, :, idx], V16[:, :, idx]
    orc.decode_attend(q16, Ks, Vs, np.full((n_seq, Hkv), len(idx)), threads=threads)
    # H2O-512: attention over 513 with logits, accumulate, keep-set per unit
    _, lse, lg = orc.decode_attend(q16, Ks, Vs, np.full((n_seq, Hkv), len(idx)),
                                   want_logits=True, threads=threads)
    sc = orc.h2o_accumulate(np.zeros((n_seq, Hkv, len(idx))), lg, lse,
                            np.full((n_seq, Hkv), len(idx)))
    for b in range(n_seq):
        for h in range(Hkv):
            orc.h2o_keep(idx.astype(np.int32), sc[b, h], T, w.n_heavy, w.n_recent)
    # KIVI-4: quantise the unit's history and attend (the oracle has no incremental state)
    g = Hq // Hkv
    n_q = orc.kivi_nq(T, w.kivi_R)
    for b in range(n_seq):
        for h in range(Hkv):
            qz = orc.kivi_quantize_unit(K16[b, h, :n_q], V16[b, h, :n_q], n_q, 4)
            orc.kivi_attend_unit(q16[b, h * g:(h + 1) * g], K16[b, h], V16[b, h], T, w.kivi_R, 4,
                                 qz=qz)
    return time.perf_counter() - t0, 4 * n_seq


def run_profile(args):
    """Small case of one kernel for ncu captures: the heavy-load workload cut to
    --profile-batch sequences (still larger than L2), one warm-up and two measured launches."""
    import torch
    import kv_cache_compression_split_gb300 as kvc
    from kv_cache_compression_split_gb300 import build as kbuild
    from kv_cache_compression_split_gb300 import workloads as W
    kbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = W.HEAVY
    B, Hq, Hkv, D, T = args.profile_batch, w.Hq, w.Hkv, w.D, w.T
    K, V = W.kv_tensors(w, T=T, B=B, device=dev)
    q = W.q_tensor(w, B=B, device=dev)
    o = torch.empty_like(q)
    what = args.profile
    if what in ("attend_fp16", "attend_h2o", "h2o_evict", "stream_evict", "h2o_acc"):
        n_slots = T if what == "attend_fp16" else 513
        cache = kvc.SlotCache.empty(B, Hkv, n_slots + 7, D, device=dev)
        kvc.kvc_append(cache, K[:, :, :n_slots].contiguous(), V[:, :, :n_slots].contiguous())
        ws = torch.empty(max(kvc.kvc_workspace_size(cache, q) // 4, 1), device=dev)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
        scores = torch.rand(B, Hkv, cache.C, device=dev)
        for _ in range(3):
            if what == "attend_h2o":   # attention + fused score update, logits on chip
                kvc.kvc_decode_attend(cache, q, o, lse=lse, num_splits=1, h2o_scores=scores)
            elif what == "h2o_acc":    # score update from logits the attention wrote to HBM
                if _ == 0:
                    logits = torch.empty(B, Hq, cache.C, device=dev)
                    kvc.kvc_decode_attend(cache, q, o, logits=logits, lse=lse, workspace=ws)
                kvc.kvc_h2o_accumulate_decode(cache, scores, logits, lse, Hq)
            elif what.startswith("attend"):
                kvc.kvc_decode_attend(cache, q, o, lse=lse, workspace=ws)
            elif what == "h2o_evict":
                c = kvc.SlotCache(cache.K, cache.V, cache.pos.clone(), cache.n.clone(), cache.seqlen)
                kvc.kvc_h2o_evict(c, scores.clone(), w.n_heavy, w.n_recent)
            else:
                c = kvc.SlotCache(cache.K, cache.V, cache.pos.clone(), cache.n.clone(), cache.seqlen)
                kvc.kvc_stream_evict(c, w.n_sink, w.n_recent)
    elif what in ("attend_kivi4", "combine"):
        # combine: the same attention forced into two splits, for the merge launch
        splits = 2 if what == "combine" else 0
        cache = kvc.QuantCache.empty(B, Hkv, T, D, 4, w.kivi_R, device=dev)
        kvc.kvc_append_quant(cache, K, V)
        del K, V   # the capture holds only what the attention reads
        torch.cuda.empty_cache()
        ws = torch.empty(max(kvc.kvc_workspace_size(cache, q, splits) // 4, 1), device=dev)
        for _ in range(3):
            kvc.kvc_decode_attend(cache, q, o, workspace=ws, num_splits=splits)
    elif what == "attend_gear4":
        cache = kvc.QuantCache.empty(B, Hkv, T, D, 4, w.kivi_R, device=dev, gear=True)
        kvc.kvc_append_quant(cache, K, V)
        del K, V
        torch.cuda.empty_cache()
        ws = torch.empty(max(kvc.kvc_workspace_size(cache, q) // 4, 1), device=dev)
        for _ in range(3):
            kvc.kvc_decode_attend(cache, q, o, workspace=ws)
    elif what in ("kivi_pack", "gear_pack"):
        for _ in range(3):
            cache = kvc.QuantCache.empty(B, Hkv, T, D, 4, w.kivi_R, device=dev,
                                         gear=what == "gear_pack")
            kvc.kvc_append_quant(cache, K, V)
    elif what == "prefill":
        L = T - 1
        qp = W.q_tensor(w, B=max(1, B // 4), L=L, device=dev)
        kp = K[:max(1, B // 4), :, :L].contiguous()
        sc = torch.zeros(kp.shape[0], Hkv, L, device=dev)
        ws = torch.empty(kvc.kvc_h2o_workspace_size(kp.shape[0], Hq, L) // 4, device=dev)
        for _ in range(3):
            kvc.kvc_h2o_accumulate_prefill(qp, kp, sc, ws, L)
    elif what == "decode_steps":
        # the benchmark's decode step (its four methods one after another) at --profile-batch
        # sequences, five times, after an untimed set-up: for a launch list of one step
        Ch = 520
        fp = kvc.SlotCache.empty(B, Hkv, T + 8, D, device=dev)
        kvc.kvc_append(fp, K[:, :, :T - 1].contiguous(), V[:, :, :T - 1].contiguous())
        h2o = kvc.SlotCache.empty(B, Hkv, Ch, D, device=dev)
        st = kvc.SlotCache.empty(B, Hkv, Ch, D, device=dev)
        for c in (h2o, st):
            kvc.kvc_append(c, K[:, :, T - 513:T - 1].contiguous(), V[:, :, T - 513:T - 1].contiguous())
            c.pos[:, :, :512] = torch.cat([torch.arange(w.n_sink),
                                           torch.arange(T - 1 - w.n_recent, T - 1)]).int().to(dev)
            c.seqlen.fill_(T - 1)
        sc = torch.rand(B, Hkv, Ch, device=dev)
        kv4 = kvc.QuantCache.empty(B, Hkv, T + 64, D, 4, w.kivi_R, device=dev)
        kvc.kvc_append_quant(kv4, K[:, :, :T - 1].contiguous(), V[:, :, :T - 1].contiguous())
        ws_fp = torch.empty(max(kvc.kvc_workspace_size(fp, q) // 4, 1), device=dev)
        ws_kv = torch.empty(max(kvc.kvc_workspace_size(kv4, q) // 4, 1), device=dev)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
        kn = torch.randn(B, Hkv, 1, D, device=dev, dtype=torch.float16)
        torch.cuda.synchronize()
        for _ in range(5):
            kvc.kvc_append(fp, kn, kn)
            kvc.kvc_decode_attend(fp, q, o, workspace=ws_fp)
            kvc.kvc_h2o_decode_step(h2o, sc, q, kn, kn, o, lse, w.n_heavy, w.n_recent)
            kvc.kvc_append_quant(kv4, kn, kn)
            kvc.kvc_decode_attend(kv4, q, o, workspace=ws_kv)
            kvc.kvc_stream_decode_step(st, q, kn, kn, o, None, w.n_sink, w.n_recent)
    elif what in ("h2o_step", "stream_step"):
        # the one-launch decode steps at the heavy-load shape: 512 slots per unit (64 sinks or
        # heavy + 448 recent), then three steps (each appends one token and keeps 512 / 513)
        cache = kvc.SlotCache.empty(B, Hkv, 520, D, device=dev)
        kvc.kvc_append(cache, K[:, :, T - 512:T].contiguous(), V[:, :, T - 512:T].contiguous())
        cache.pos[:, :, :512] = torch.cat([torch.arange(w.n_sink),
                                           torch.arange(T - w.n_recent, T)]).int().to(dev)
        cache.seqlen.fill_(T)
        sc = torch.rand(B, Hkv, 520, device=dev)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
        kn = torch.randn(B, Hkv, 1, D, device=dev, dtype=torch.float16)
        for _ in range(3):
            if what == "h2o_step":
                kvc.kvc_h2o_decode_step(cache, sc, q, kn, kn, o, lse, w.n_heavy, w.n_recent)
            else:
                kvc.kvc_stream_decode_step(cache, q, kn, kn, o, None, w.n_sink, w.n_recent)
    elif what == "stream_append":
        # the heavy-load StreamingLLM-512 decode append: 512 slots of sinks + recent window,
        # then three one-token appends (the first grows the window to 513, the next two
        # overwrite the slot of the token that leaves it)
        cache = kvc.SlotCache.empty(B, Hkv, 520, D, device=dev)
        kvc.kvc_append(cache, K[:, :, :T - 1].contiguous()[:, :, :512].contiguous(),
                       V[:, :, :512].contiguous())
        cache.pos[:, :, :512] = torch.cat([torch.arange(w.n_sink),
                                           torch.arange(T - 1 - w.n_recent, T - 1)]).int().to(dev)
        cache.seqlen.fill_(T - 1)
        for i in range(3):
            kvc.kvc_stream_append(cache, K[:, :, T - 1 + i - 2:T - 1 + i - 1].contiguous(),
                                  V[:, :, T - 1 + i - 2:T - 1 + i - 1].contiguous(), w.n_sink,
                                  w.n_recent)
    elif what == "random_evict":
        # reasoning-trace steady state (epoch 30): 1024 locked prompt tokens, 341 kept earlier
        # tokens, 1024 new ones -> 1365 per head after the eviction; --profile-batch sequences
        wr = W.REASONING
        n0, P = 1024 + 341 + 1024, wr.prompt_len
        Kr, Vr = W.kv_tensors(wr, T=n0, B=B, device=dev)
        cache = kvc.SlotCache.empty(B, wr.Hkv, 2432, wr.D, device=dev)
        kvc.kvc_append(cache, Kr, Vr)
        gp = torch.Generator().manual_seed(30)
        old = torch.randperm(31744 - P, generator=gp)[:341].sort().values + P
        posr = torch.cat([torch.arange(P), old, torch.arange(31744, 32768)]).int().to(dev)
        cache.pos[:, :, :n0] = posr
        cache.seqlen.fill_(32768)
        pos0 = cache.pos.clone()
        for _ in range(3):
            cache.pos.copy_(pos0)
            cache.n.fill_(n0)
            kvc.kvc_random_evict(cache, P, wr.keep_ratio, W.RANDOM_EVICT_SEED, 30)
    elif what in ("attend_kivi2_mha", "attend_kivi4_mha"):
        # the KIVI workload: 32 MHA heads, T = 4096, offsets on Q, K, V; --profile-batch sequences
        wk = W.KIVI_MHA
        bits = 2 if what == "attend_kivi2_mha" else 4
        Kk, Vk = W.kv_tensors(wk, T=wk.T, B=B, device=dev)
        qk = W.q_tensor(wk, B=B, device=dev)
        ok = torch.empty_like(qk)
        cache = kvc.QuantCache.empty(B, wk.Hkv, wk.T, wk.D, bits, wk.kivi_R, device=dev)
        kvc.kvc_append_quant(cache, Kk, Vk)
        del Kk, Vk
        torch.cuda.empty_cache()
        ws = torch.empty(max(kvc.kvc_workspace_size(cache, qk) // 4, 1), device=dev)
        for _ in range(3):
            kvc.kvc_decode_attend(cache, qk, ok, workspace=ws)
    elif what in ("kivi_append_flush", "gear_append_flush"):
        # decode-sized append whose token completes a group: the bulk pack of 2047 tokens
        # (two launches), then three one-token appends from length 2047, each flushing group 59
        cache = kvc.QuantCache.empty(B, Hkv, T + 32, D, 4, w.kivi_R, device=dev,
                                     gear=what == "gear_append_flush")
        kvc.kvc_append_quant(cache, K[:, :, :T - 1].contiguous(), V[:, :, :T - 1].contiguous())
        kn, vn = K[:, :, T - 1:T].contiguous(), V[:, :, T - 1:T].contiguous()
        for _ in range(3):
            cache.len.fill_(T - 1)
            kvc.kvc_append_quant(cache, kn, vn)
    else:
        raise SystemExit(f"unknown --profile {what}")
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status() == 0
    print(f"profile case {what}: ok")


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    import oracle as orc
    orc.build()
    threads = cpu_cores()
    n_seq = args.ref_seqs
    for _ in range(args.warmup):
        oracle_sample(max(1, n_seq // 4), threads)
    times, toks = [], 0
    for _ in range(args.steps):
        dt, tk = oracle_sample(n_seq, threads)
        times.append(dt)
        toks += tk
    value = toks / sum(times)
    sample = (f"{n_seq} sequences x 8 KV heads of the heavy-load workload per step, one decode "
              f"step of FP16, StreamingLLM-512, H2O-512 and KIVI-4 (oracle, fp64)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "heavy-gqa64x8-b512-d128-t2048", "global_batch": n_seq,
                       "seq_len": 2048, "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_grid(args):
    """Throughput profile grid: batch x KV length x method on the heavy-load head layout (GQA 64/8,
    D 128), the per-method cost table a router consumes.  Per (B, T) cell and method:
      prefill_ms  compress a T-token prompt: FP16 append; KIVI-b / GEAR-4 pack; StreamingLLM and H2O evict
                  to 64 + 448 (H2O after its two-pass score pass); random eviction at each keep
                  ratio with the first min(1024, T/2) tokens locked
      decode_ms   one decode step over the cache the prefill left: FP16 and KIVI append +
                  attention; H2O and StreamingLLM one launch each (kvc_h2o_decode_step,
                  kvc_stream_decode_step); for random eviction, attention over the kept slots
    Every timing is the median of 3 repetitions after one warm-up, with L2 flushed (a 512 MB
    write, then a 512 MB read) before each; one JSON line per cell."""
    import torch
    import kv_cache_compression_split_gb300 as kvc
    from kv_cache_compression_split_gb300 import build as kbuild
    kbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    Hq, Hkv, D, R = 64, 8, 128, 128
    n_heavy, n_recent, n_sink = 64, 448, 64
    ratios = [1.0, 0.75, 0.5, 0.25, 0.125]
    batches = [int(x) for x in args.grid_batches.split(",")]
    lengths = [int(x) for x in args.grid_lengths.split(",")]
    flush = L2Flush(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, setup=None, reps=3):
        ts = []
        for r in range(reps + 1):
            if setup is not None:
                setup()
            flush()
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if r > 0:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    def ws_for(cache, q, splits=0):
        nb = kvc.kvc_workspace_size(cache, q, splits)
        return torch.empty(max(nb // 4, 1), dtype=torch.float32, device=dev)

    for B in batches:
        for T in lengths:
            cell = {"B": B, "T": T, "heads": f"GQA {Hq}/{Hkv}", "D": D, "prefill_ms": {},
                    "decode_ms": {}, "decode_tokens_per_s": {}, "slots_attended": {}}
            with torch.cuda.stream(stream):
                gen = torch.Generator(device=dev)
                gen.manual_seed(1000 + B + T)
                K = torch.randn(B, Hkv, T, D, generator=gen, device=dev, dtype=torch.float16)
                V = torch.randn(B, Hkv, T, D, generator=gen, device=dev, dtype=torch.float16)
                q = torch.randn(B, Hq, D, generator=gen, device=dev, dtype=torch.float16)
                kn = torch.randn(B, Hkv, 1, D, generator=gen, device=dev, dtype=torch.float16)
                vn = torch.randn(B, Hkv, 1, D, generator=gen, device=dev, dtype=torch.float16)
                o = torch.empty_like(q)
                C = T + 8
                fp = kvc.SlotCache.empty(B, Hkv, C, D, device=dev)

                def small_cache(src, Cs=520):
                    # the first Cs slots of an evicted cache as a decode cache of capacity Cs
                    c = kvc.SlotCache.empty(B, Hkv, Cs, D, device=dev)
                    m = min(Cs, src.C)
                    c.K[:, :, :m] = src.K[:, :, :m]
                    c.V[:, :, :m] = src.V[:, :, :m]
                    c.pos[:, :, :m] = src.pos[:, :, :m]
                    c.n.copy_(src.n)
                    c.seqlen.copy_(src.seqlen)
                    return c

                def refill():
                    fp.n.zero_()
                    fp.seqlen.zero_()
                    kvc.kvc_append(fp, K, V, stream=stream)

                def rewind(n):
                    fp.n.fill_(n)
                    fp.seqlen.fill_(n)

                # ---- FP16
                cell["prefill_ms"]["fp16"] = timed(lambda: kvc.kvc_append(fp, K, V, stream=stream),
                                                   setup=lambda: rewind(0))
                ws = ws_for(fp, q)

                def fp_step():
                    kvc.kvc_append(fp, kn, vn, stream=stream)
                    kvc.kvc_decode_attend(fp, q, o, workspace=ws, stream=stream)
                cell["decode_ms"]["fp16"] = timed(fp_step, setup=lambda: rewind(T))
                cell["slots_attended"]["fp16"] = T + 1
                # ---- random eviction sweep (prompt locked), attention over the kept slots
                prompt = min(1024, T // 2)
                for r in ratios:
                    name = f"random{r:g}"
                    cell["prefill_ms"][name] = timed(
                        lambda: kvc.kvc_random_evict(fp, prompt, r, 0x243F6A8885A308D3, 0,
                                                     stream=stream), setup=refill)
                    kept = prompt + max(1, int((T - prompt) * r))
                    cell["decode_ms"][name] = timed(
                        lambda: kvc.kvc_decode_attend(fp, q, o, workspace=ws, stream=stream))
                    cell["slots_attended"][name] = kept
                # ---- StreamingLLM: evict the prompt to 64 sinks + 448 recent, then steady steps
                cell["prefill_ms"]["stream512"] = timed(
                    lambda: kvc.kvc_stream_evict(fp, n_sink, n_recent, stream=stream), setup=refill)
                # the decode cache: the kept window in a 520-slot cache, one-launch steps
                st = small_cache(fp)

                def stream_step():
                    kvc.kvc_stream_decode_step(st, q, kn, vn, o, None, n_sink, n_recent,
                                               stream=stream)
                cell["decode_ms"]["stream512"] = timed(stream_step)
                cell["slots_attended"]["stream512"] = n_sink + n_recent + 1
                del st
                # ---- H2O: two-pass prefill score pass (in batch chunks of <= 8 GB of queries)
                # then evict to 64 heavy + 448 recent; decode steps with the fused update
                scores = torch.zeros(B, Hkv, C, dtype=torch.float32, device=dev)
                bc = max(1, min(B, (8 << 30) // (Hq * T * D * 2)))
                qp = torch.randn(bc, Hq, T, D, generator=gen, device=dev, dtype=torch.float16)
                pws = torch.empty(kvc.kvc_h2o_workspace_size(bc, Hq, T) // 4, dtype=torch.float32,
                                  device=dev)

                def h2o_prefill():
                    for b0 in range(0, B, bc):
                        b1 = min(B, b0 + bc)
                        kvc.kvc_h2o_accumulate_prefill(qp[:b1 - b0], fp.K[b0:b1], scores[b0:b1],
                                                       pws, T, stream=stream)
                    kvc.kvc_h2o_evict(fp, scores, n_heavy, n_recent, stream=stream)
                cell["prefill_ms"]["h2o512"] = timed(h2o_prefill, setup=refill, reps=1)
                del qp, pws
                lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
                hc = small_cache(fp)
                hsc = torch.zeros(B, Hkv, 520, dtype=torch.float32, device=dev)
                hsc[:, :, :min(520, C)] = scores[:, :, :min(520, C)]

                def h2o_step():
                    kvc.kvc_h2o_decode_step(hc, hsc, q, kn, vn, o, lse, n_heavy, n_recent,
                                            stream=stream)
                cell["decode_ms"]["h2o512"] = timed(h2o_step)
                cell["slots_attended"]["h2o512"] = n_heavy + n_recent + 1
                del fp, scores, lse, hc, hsc
                # ---- KIVI-4 / KIVI-2 / GEAR-4: pack the prompt, then append + attention
                for bits, gear in ((4, False), (2, False), (4, True)):
                    name = f"gear{bits}" if gear else f"kivi{bits}"
                    kv = kvc.QuantCache.empty(B, Hkv, 32 * ((T + 1) // 32 + 1), D, bits, R,
                                              device=dev, gear=gear)
                    cell["prefill_ms"][name] = timed(
                        lambda: kvc.kvc_append_quant(kv, K, V, stream=stream),
                        setup=lambda: kv.len.zero_())
                    ws_k = ws_for(kv, q)

                    def kivi_step():
                        kvc.kvc_append_quant(kv, kn, vn, stream=stream)
                        kvc.kvc_decode_attend(kv, q, o, workspace=ws_k, stream=stream)
                    cell["decode_ms"][name] = timed(kivi_step, setup=lambda: kv.len.fill_(T))
                    cell["slots_attended"][name] = T + 1
                    del kv, ws_k
                del K, V
            torch.cuda.synchronize(dev)
            status = kvc.kvc_read_device_status(stream)
            cell["device_status"] = status
            cell["decode_tokens_per_s"] = {k: B / (v * 1e-3) for k, v in cell["decode_ms"].items()}
            print(json.dumps(cell), flush=True)
            torch.cuda.empty_cache()


def max_over_ranks(values, world: int, device):
    """Per-rank timings reduced with MAX over all ranks (every rank gets the result)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world: int, tokens_per_step_per_rank: int, ms_per_step: float) -> float:
    """Tokens/s of the whole job: every rank processes its own batch (weak scaling) and the
    step time is the slowest rank's."""
    return world * tokens_per_step_per_rank / (ms_per_step * 1e-3)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--ref-seqs", type=int, default=4)
    ap.add_argument("--cpu-seqs", type=int, default=24)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", default=None,
                    help="run one kernel on a small case for ncu: attend_fp16, attend_h2o, "
                         "attend_kivi4, attend_gear4, attend_kivi2_mha, attend_kivi4_mha, "
                         "h2o_evict, stream_evict, stream_append, random_evict, prefill, h2o_acc, "
                         "kivi_pack, gear_pack, kivi_append_flush, gear_append_flush, "
                         "combine (KIVI-4 attention in two splits and their merge)")
    ap.add_argument("--profile-batch", type=int, default=64)
    ap.add_argument("--grid", action="store_true",
                    help="throughput profile grid over batch x KV length x method (JSON lines)")
    ap.add_argument("--grid-batches", default="1,16,128,512")
    ap.add_argument("--grid-lengths", default="1024,4096,16384")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.profile:
        run_profile(args)
        return
    if args.grid:
        run_grid(args)
        return
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    # the CPU baseline (oracle) runs first, before any CUDA context exists
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle as orc
        orc.build()
        threads = cpu_cores()
        dt, tk = oracle_sample(args.cpu_seqs, threads)
        dt1, tk1 = oracle_sample(2, 1)   # the same work per sequence on one core
        dtp = oracle_prefill_sample(2, threads)
        cpu = {"value": tk / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
               "value_1_core": tk1 / dt1,
               "prefill_s_extrapolated": dtp * 512 / 2,
               "prefill_sample": "H2O prefill score pass of 2 sequences (2047-token prompt, "
                                 f"8 KV heads) in {dtp:.1f} s on {threads} threads, scaled "
                                 "linearly to the 512 sequences of the GPU row",
               "sample": f"{args.cpu_seqs} sequences x 8 KV heads of the heavy-load workload, one "
                         f"decode step of FP16, StreamingLLM-512, H2O-512 and KIVI-4 "
                         f"({dt:.1f} s of fp64 oracle work); value_1_core: 2 sequences on one "
                         f"thread ({dt1:.1f} s)"}

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_gpu(args, rank, world)
    ms, e2e_ms = max_over_ranks([res["ms_per_step"], res["e2e_ms_per_step"]], world, "cuda")
    if rank == 0:
        dom = res["kernels"]["attend_fp16"]
        line = {
            "metric": METRIC, "value": whole_job_rate(world, res["tokens_per_step"], ms),
            "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": "heavy-gqa64x8-b512-d128-t2048", "global_batch": 512 * world,
                       "seq_len": 2048, "parallelism": f"replicas x{world}",
                       "methods": ["fp16", "h2o512", "kivi4", "stream512"],
                       "kv_len": "2048 + step index (each step appends one token)",
                       "l2": "inputs larger than L2 (8 GB of cache read per step)",
                       "launch": "the timed steps captured in one CUDA graph, launched once; "
                                 "each step runs the four methods on four streams (fork/join "
                                 "per step)"},
            "e2e": {"value": whole_job_rate(world, res["tokens_per_step"], e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                    "ms_per_step_replays": res["e2e_runs_ms"],
                    "host_binding": res["host_binding"]},
            "gpu_launches": res["launches_per_step"] * args.steps,
            "roofline": {"bound": "hbm", "kernel": "k_attend_slots (FP16 cache launch)",
                         "achieved": dom["gbs"], "peak": res["hbm_peak"], "unit": "GB/s",
                         "frac": dom["frac_of_hbm"], "traffic": res["fp16_traffic"],
                         "algorithmic_bytes": dom["bytes_per_step"],
                         "peak_source": res["peak_kind"],
                         # the compressed decode-attention launches of the same step
                         "compressed": {
                             nm: {"kernel": kn_, "achieved": res["kernels"][k]["gbs"],
                                  "frac": res["kernels"][k]["frac_of_hbm"],
                                  "algorithmic_bytes": res["kernels"][k]["bytes_per_step"]}
                             for nm, k, kn_ in (
                                 ("h2o512", "attend_h2o512",
                                  "k_attend_slots decode step (H2O-512: append, attention, "
                                  "score update, eviction)"),
                                 ("stream512", "attend_stream512",
                                  "k_attend_slots decode step (Stream-512: append, attention)"),
                                 ("kivi4", "attend_kivi4", "k_attend_kivi (KIVI-4)"))}},
            "cpu_baseline": cpu,
            "clocks": res["clocks"],
            "kernels": res["kernels"], "methods": res["methods"], "rows": res["rows"],
            "calls_ms": res["calls_ms"], "eager_ms_per_step": res["eager_ms_per_step"],
            "serial_ms_per_step": res["serial_ms_per_step"],
            "step_roofline": res["step_roofline"],
            "device_status": res["device_status"],
            "kivi_window": res["kivi_window"],
        }
        print(json.dumps(line))


if __name__ == "__main__":
    main()
