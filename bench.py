#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300: chunked prefill + decode step.

One step = one kda_chunk_prefill over a 145408-token prompt (H=32, Dk=Dv=128,
fp32 initial state, checkpoints every 32768 tokens and at the end: 5 per head)
followed by one kda_decode_step over 512 sequences x 32 heads (1.07 GB of fp32
state updated in place).  Inputs are seeded synthetic tensors with the
shapes and value distributions of the workloads (see workloads.py), resident
in HBM and larger than the 129 MB L2, so no L2 flush is needed between steps.

`value` = prefill tokens/s (whole job: tokens of all ranks / max-over-ranks
time).  The decode step's state-update bandwidth is reported alongside.

With N > 1 ranks (one per GPU), --split chooses what a rank serves:
  replicas (default)  its own prompt and decode batch: weak scaling;
  heads               H / N heads of the one prompt and of the one decode batch:
                      strong scaling.  KDA heads are independent recurrences, so
                      neither split has a collective on the data path.  With few
                      heads per rank the prompt's chunks are split too
                      (kda_chunk_prefill_segmented; --segments auto|P).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--split replicas|heads]

--impl reference times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload), the reference arm for this method.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (T=142k, H=32, D=128) + decode state-update HBM GB/s"
T_PROMPT, H, D, CKPT = 145408, 32, 128, 32768
DEC_N = 512
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0

# Algorithmic bytes: per token per head q, k, v bf16
# (3 x 256 B), log_alpha fp32 (512 B), beta bf16 (2 B), o bf16 (256 B).
BYTES_PER_TOKEN_HEAD = 3 * 2 * D + 4 * D + 2 + 2 * D           # 1538
STATE_BYTES = 4 * D * D                                          # one fp32 head state
# Useful FLOPs: the FlashKDA count 12C^3 + 8C^2 D + 6 C D^2 per 64-token chunk per head.
FLOPS_PER_CHUNK = 12 * 64 ** 3 + 8 * 64 ** 2 * D + 6 * 64 * D ** 2


def prefill_algorithmic_bytes(T, n_ckpt_per_head, heads=H):
    # inputs + output, plus init-state read, final-state write and checkpoint writes
    return BYTES_PER_TOKEN_HEAD * T * heads + STATE_BYTES * heads * (2 + n_ckpt_per_head)


def kv_state_bytes(n_ckpt_per_head, heads=H):
    """Bytes of recurrent state one prefill hands to a prefix cache: the final state and
    every checkpoint, all heads (the 'KV size' of KV throughput = KV size / prefill time)."""
    return STATE_BYTES * heads * (1 + n_ckpt_per_head)


def decode_algorithmic_bytes(N, heads=H):
    # state read + write, plus q, k, v, log_alpha, beta in and o out
    return N * heads * (2 * STATE_BYTES + BYTES_PER_TOKEN_HEAD)


def reduce_max(values, device="cpu"):
    """Element-wise max of a list of floats over all ranks (identity on one process)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(units_per_rank, world, slowest_ms):
    """Weak-scaling throughput: every rank processes units_per_rank in parallel; the job
    takes as long as the slowest rank."""
    return units_per_rank * world / (slowest_ms / 1e3)


def rank_seed(base, rank):
    """Each rank serves its own prompt and decode batch (independent problems)."""
    return base + 1000 * rank


def head_range(h_total, world, rank):
    """Heads [h0, h1) of rank `rank` when one problem's h_total heads are split evenly
    over `world` ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if h_total % world:
        raise ValueError(f"{h_total} heads do not split evenly over {world} ranks")
    n = h_total // world
    return rank * n, (rank + 1) * n


def job_rate(units, world, slowest_ms, split):
    """Whole-job throughput.  replicas: every rank processes `units` of its own (weak
    scaling); heads: the ranks process one set of `units` between them (strong scaling).
    Either way the job takes as long as the slowest rank."""
    if split not in ("replicas", "heads"):
        raise ValueError(split)
    return whole_job_rate(units, world if split == "replicas" else 1, slowest_ms)


def rank_problem(split, world, rank):
    """(heads served, seed offset) of a rank: replicas draw their own problems from
    per-rank seeds; a head split cuts the one problem (seed offset 0) into head ranges."""
    if split == "heads":
        return head_range(H, world, rank), 0
    return (0, H), 1000 * rank


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        hbm = d.get("hbm_gbs") or d.get("hbm_GBps") or d.get("hbm")
        bf = d.get("bf16_tflops")
        bfs = d.get("bf16_tflops_sustained")
        if hbm:
            return float(hbm), float(bf or FALLBACK_BF16_TFLOPS), float(bfs or bf or FALLBACK_BF16_TFLOPS), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def read_traffic(kernel):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    kernel source that is built now (source hash recorded beside the figure)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f).get(kernel)
        if not d:
            return None
        src = os.path.join(ROOT, "kimi_delta_attention_06_gb300", "csrc", d["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return float(d["bytes_per_launch"]) if h == d["source_sha256_16"] else None
    except (OSError, ValueError, KeyError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi sampling during the timed region (SM clock, throttle reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t_lo, t_hi = getattr(self, "t_start", 0.0), getattr(self, "t_stop", float("inf"))
        inside = [ln for (ts, ln) in self.lines if t_lo <= ts <= t_hi]
        for ln in inside or [ln for (_, ln) in self.lines]:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1])); smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_count():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(budget_s=12.0):
    """Time the fp64 oracle on a bounded sample of the same workload: all 32 heads of
    the first n tokens of the 145408-token prompt, plus a decode step on a subset of
    the 512 sequences.  n grows until the prefill sample takes about budget_s/2."""
    import torch
    import oracle
    from kimi_delta_attention_06_gb300 import workloads
    oracle.build()
    threads = cpu_count()
    n = 256
    res = None
    while True:
        c = workloads.single_case(n, seed=2)
        t0 = time.perf_counter()
        oracle.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, c.init_state, threads=threads)
        dt = time.perf_counter() - t0
        res = (n, dt)
        if dt > budget_s / 2 or n >= T_PROMPT:
            break
        n = min(T_PROMPT, int(n * max(2.0, min(16.0, (budget_s / 2) / max(dt, 1e-3)))))
    n_tok, dt = res
    pre_tps = n_tok / dt
    nd = 64
    dc = workloads.decode_case(N=nd, H=H, D=D, steps=1, seed=4)
    s = dc.steps[0]
    t0 = time.perf_counter()
    oracle.decode(s["q"], s["k"], s["v"], s["log_alpha"], s["beta"], dc.state, threads=threads)
    ddt = time.perf_counter() - t0
    dec_gbs = decode_algorithmic_bytes(nd) / ddt / 1e9
    return {"value": pre_tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"prefill: first {n_tok} tokens x {H} heads of the {T_PROMPT}-token prompt "
                      f"({dt:.2f} s); decode: {nd} of {DEC_N} sequences x {H} heads ({ddt:.2f} s)",
            "decode_gbs": dec_gbs, "prefill_seconds": dt}


def time_module_path(dev, stream, heads=(0, H), seed_offset=0, steps=10):
    """The KDA module around the recurrence at T=145408, H=32, D=128, timed on the device:
    kda_prepare_inputs (short conv + SiLU, L2 norm of q and k, alpha and beta gates) then
    kda_chunk_prefill_ex with the per-head output norm fused into its output epilogue: two
    launches per step.  The three-pass form (prepare, prefill, kda_output_norm) is timed
    beside it; both write the same normed bf16 output."""
    import torch
    from kimi_delta_attention_06_gb300 import kda, workloads
    m = workloads.module_case(T_PROMPT, H=H, D=D, seed=5 + seed_offset, device=dev)
    Hl = heads[1] - heads[0]
    if Hl != H:
        m = workloads.head_slice(m, *heads)
    cu = m.cu_seqlens.to(dev)
    q, k, v = (torch.empty(T_PROMPT, Hl, D, device=dev, dtype=torch.bfloat16) for _ in range(3))
    la = torch.empty(T_PROMPT, Hl, D, device=dev)
    beta = torch.empty(T_PROMPT, Hl, device=dev, dtype=torch.bfloat16)
    s0 = torch.zeros(1, Hl, D, D, device=dev)
    o = torch.empty(T_PROMPT, Hl, D, device=dev, dtype=torch.bfloat16)
    y = torch.empty_like(o)
    fin = torch.empty(1, Hl, D, D, device=dev)

    def prepare():
        kda.kda_prepare_inputs(m.xq, m.xk, m.xv, m.conv_w, None, m.a_raw, m.b_raw, cu, m.cu_seqlens, 1, T_PROMPT,
                               Hl, D, 1, q, k, v, la, beta, stream)

    def prefill(norm):
        kda.kda_chunk_prefill_ex(q, k, v, la, beta, s0, cu, m.cu_seqlens, 1, T_PROMPT, Hl, D, D, y if norm else o,
                                 kda.KDA_OUT_BF16, fin, None, 0, kda.KDA_DECAY_CHANNEL,
                                 out_norm_gamma=m.gamma if norm else None, out_norm_eps=1e-6, stream=stream)

    def norm():
        kda.kda_output_norm(o, kda.KDA_OUT_BF16, m.gamma, 1e-6, y, T_PROMPT, Hl, D, stream)

    res = {}
    for name, parts in (("fused", [prepare, lambda: prefill(True)]),
                        ("separate", [prepare, lambda: prefill(False), norm])):
        for _ in range(3):
            for f in parts:
                f()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            ev[i][0].record(stream)
            for j, f in enumerate(parts):
                f()
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize()
        per = [statistics.median(e[j].elapsed_time(e[j + 1]) for e in ev) for j in range(len(parts))]
        tot = statistics.median(e[0].elapsed_time(e[-1]) for e in ev)
        res[name] = {"ms_per_step": tot, "launch_ms": per, "tokens_per_s": T_PROMPT / (tot / 1e3),
                     "heads": Hl}
    if kda.kda_device_status() != 0:
        raise RuntimeError("device status after the module path")
    res["workload"] = (f"prepare (conv width 4 + SiLU, L2 norm, gates) -> prefill T={T_PROMPT} H={Hl} Dk=Dv={D} "
                       f"-> per-head output norm; zero initial state, no checkpoints")
    res["launches"] = {"fused": ["kda_prepare_inputs", "kda_chunk_prefill_ex (+norm)"],
                       "separate": ["kda_prepare_inputs", "kda_chunk_prefill_ex", "kda_output_norm"]}
    return res


def _median_ms(fns, stream, steps):
    """Median CUDA-event time of `fns` run back to back, after 3 untimed rounds."""
    import torch
    for _ in range(3):
        for f in fns:
            f()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        for f in fns:
            f()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def time_other_rows(dev, stream, heads=(0, H), seed_offset=0, steps=10):
    """The workloads beside the headline, timed on the device after the main timed region:
    - varlen: 16 packed sequences of log-uniform length in [1k, 64k] (279,375 tokens), even
      ones from an initial state, checkpoints every 32768 tokens; and the same pack on 2
      heads, plain and segmented;
    - layouts: the T=145408 prompt with one decay per head (Gated DeltaNet) and with none
      (DeltaNet), through kda_chunk_prefill_ex;
    - serving decode: kda_decode_multi over a 512-slot x H state pool, K = 8 tokens per
      sequence, verify (states untouched) and commit (states written back)."""
    import torch
    from kimi_delta_attention_06_gb300 import kda, workloads
    h0, h1 = heads
    Hl = h1 - h0
    res = {}

    def cut(case):
        return case if Hl == H else workloads.head_slice(case, h0, h1)

    vc = cut(workloads.varlen_case(seed=3 + seed_offset, device=dev, H=H, D=D, ckpt_stride=CKPT))
    cu = vc.cu_seqlens.to(dev)
    out = torch.empty(vc.T, Hl, D, device=dev, dtype=torch.bfloat16)
    fin = torch.empty(vc.N, Hl, D, D, device=dev)
    nck = kda.kda_ckpt_count(vc.cu_seqlens, CKPT)
    ck = torch.empty(max(nck, 1), Hl, D, D, device=dev)
    ms = _median_ms([lambda: kda.kda_chunk_prefill(vc.q, vc.k, vc.v, vc.log_alpha, vc.beta, vc.init_state, cu,
                                                   vc.cu_seqlens, vc.N, vc.T, Hl, D, D, out, kda.KDA_OUT_BF16, fin,
                                                   ck if nck else None, CKPT, stream)], stream, steps)
    res["varlen"] = {"ms": ms, "tokens": vc.T, "sequences": vc.N, "tokens_per_s": vc.T / (ms / 1e3),
                     "workload": vc.name}
    # the same pack on 2 heads (one GPU's share of a 32-head model over 16 GPUs): plain
    # against segmented (kda_chunk_prefill_segmented_ex)
    if Hl >= 2:
        v2 = workloads.head_slice(vc, 0, 2)
        o2 = torch.empty(v2.T, 2, D, device=dev, dtype=torch.bfloat16)
        f2 = torch.empty(v2.N, 2, D, D, device=dev)
        k2 = torch.empty(max(nck, 1), 2, D, D, device=dev)
        p2 = kda.segments_for(2, num_seqs=v2.N)
        plain = _median_ms([lambda: kda.kda_chunk_prefill(v2.q, v2.k, v2.v, v2.log_alpha, v2.beta, v2.init_state, cu,
                                                          v2.cu_seqlens, v2.N, v2.T, 2, D, D, o2, kda.KDA_OUT_BF16,
                                                          f2, k2 if nck else None, CKPT, stream)], stream, steps)
        segd = _median_ms([lambda: kda.kda_chunk_prefill_segmented_ex(v2.q, v2.k, v2.v, v2.log_alpha, v2.beta,
                                                                      v2.init_state, v2.cu_seqlens, v2.N, v2.T, 2, D,
                                                                      D, o2, kda.KDA_OUT_BF16, f2,
                                                                      k2 if nck else None, CKPT,
                                                                      kda.KDA_DECAY_CHANNEL, None, p2,
                                                                      stream=stream)], stream, steps)
        res["segmented_varlen_2_heads"] = {"plain_ms": plain, "segmented_ms": segd, "segments": p2,
                                           "tokens_per_s": v2.T / (segd / 1e3),
                                           "workload": f"{vc.name} heads 0-1, ckpt every {CKPT}"}
        del v2, o2, f2, k2
    del vc, out, fin, ck

    c = cut(workloads.single_case(T_PROMPT, seed=2 + seed_offset, device=dev, ckpt_stride=CKPT))
    cu = c.cu_seqlens.to(dev)
    out = torch.empty(T_PROMPT, Hl, D, device=dev, dtype=torch.bfloat16)
    fin = torch.empty(1, Hl, D, D, device=dev)
    lay = {}
    for name, decay, la in (("gated_deltanet", kda.KDA_DECAY_HEAD, c.log_alpha[:, :, 0].contiguous()),
                            ("deltanet", kda.KDA_DECAY_NONE, None)):
        ms = _median_ms([lambda: kda.kda_chunk_prefill_ex(c.q, c.k, c.v, la, c.beta, c.init_state, cu, c.cu_seqlens,
                                                          1, T_PROMPT, Hl, D, D, out, kda.KDA_OUT_BF16, fin, None,
                                                          0, decay, stream=stream)], stream, steps)
        lay[name] = {"ms": ms, "tokens_per_s": T_PROMPT / (ms / 1e3)}
    res["layouts"] = lay
    # one GPU's share of the prompt when 32 heads are split over 8 GPUs: 4 heads, plain
    # against segmented (the chain of each head is serial, so 4 heads alone leave most
    # SMs idle)
    if Hl >= 4:
        c4 = workloads.head_slice(c, 0, 4)
        nck = kda.kda_ckpt_count(c4.cu_seqlens, CKPT)
        o4 = torch.empty(T_PROMPT, 4, D, device=dev, dtype=torch.bfloat16)
        f4 = torch.empty(1, 4, D, D, device=dev)
        k4 = torch.empty(nck, 4, D, D, device=dev)
        p4 = kda.segments_for(4)
        plain = _median_ms([lambda: kda.kda_chunk_prefill(c4.q, c4.k, c4.v, c4.log_alpha, c4.beta, c4.init_state, cu,
                                                          c4.cu_seqlens, 1, T_PROMPT, 4, D, D, o4, kda.KDA_OUT_BF16,
                                                          f4, k4, CKPT, stream)], stream, steps)
        segd = _median_ms([lambda: kda.kda_chunk_prefill_segmented(c4.q, c4.k, c4.v, c4.log_alpha, c4.beta,
                                                                   c4.init_state, T_PROMPT, 4, D, D, o4,
                                                                   kda.KDA_OUT_BF16, f4, k4, CKPT,
                                                                   kda.KDA_DECAY_CHANNEL, 0, p4, stream=stream)],
                          stream, steps)
        res["segmented_4_heads"] = {"plain_ms": plain, "segmented_ms": segd, "segments": p4,
                                    "tokens_per_s": T_PROMPT / (segd / 1e3),
                                    "workload": f"prefill T={T_PROMPT} H=4 D={D} ckpt every {CKPT}"}
        del c4, o4, f4, k4
    del c, out, fin

    K = 8
    d = cut(workloads.decode_case(N=DEC_N, H=H, D=D, steps=K, seed=4 + seed_offset, device=dev))
    tok = {key: torch.stack([st[key] for st in d.steps], dim=1).contiguous()
           for key in ("q", "k", "v", "log_alpha", "beta")}
    dout = torch.empty(DEC_N, K, Hl, D, device=dev, dtype=torch.bfloat16)
    sd = {}
    for name, commit in (("verify", 0), ("commit", 1)):
        ms = _median_ms([lambda: kda.kda_decode_multi(tok["q"], tok["k"], tok["v"], tok["log_alpha"], tok["beta"],
                                                      d.state, DEC_N, None, None, commit, dout, kda.KDA_OUT_BF16,
                                                      DEC_N, K, Hl, D, D, stream=stream)], stream, steps)
        sd[name + "_ms"] = ms
    sd.update({"sequences": DEC_N, "tokens_per_sequence": K,
               "verify_tokens_per_s": DEC_N * K / (sd["verify_ms"] / 1e3)})
    res["serving_decode"] = sd
    if kda.kda_device_status() != 0:
        raise RuntimeError("device status after the other rows")
    return res


def bench_config(world, split="replicas"):
    """The workload description both arms print (the reference arm times a bounded sample of it)."""
    par = f"replicas x{world}" if split == "replicas" else f"heads split over {world} ranks ({H // world} per rank)"
    return {"workload": f"kda prefill T={T_PROMPT} H={H} Dk=Dv={D} ckpt every {CKPT} + decode N={DEC_N} H={H} D={D}",
            "global_batch": world if split == "replicas" else 1, "seq_len": T_PROMPT, "heads": H, "head_dim": D,
            "ckpt_stride": CKPT, "decode_batch": DEC_N,
            "l2": "inputs larger than L2 (no flush needed)", "parallelism": par}


def run_reference(args, rank):
    if rank != 0:
        return 0
    samples = []
    for i in range(args.warmup + args.steps):
        r = time_oracle(budget_s=max(2.0, 60.0 / max(1, args.steps + args.warmup)))
        if i >= args.warmup:
            samples.append(r)
    v = statistics.median(x["value"] for x in samples)
    cb = dict(samples[-1])
    cb["value"] = v
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(x["prefill_seconds"] for x in samples),
            "higher_is_better": True, "scaling": "weak" if args.split == "replicas" else "strong",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": bench_config(args.gpus, args.split),
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-module", action="store_true")
    ap.add_argument("--no-other", action="store_true", help="skip the varlen, layout and serving-decode rows")
    ap.add_argument("--split", choices=["replicas", "heads"], default="replicas",
                    help="N > 1: each rank serves its own problem (replicas) or H/N heads of one (heads)")
    ap.add_argument("--segments", default="auto",
                    help="prefill segments per prompt: auto (fill the GPU when a rank holds few heads) or P")
    args = ap.parse_args(argv)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank)

    import torch
    import torch.distributed as dist
    from kimi_delta_attention_06_gb300 import build as kbuild
    from kimi_delta_attention_06_gb300 import kda, workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    kbuild.build()
    kda.load()
    stream = torch.cuda.current_stream()

    # ---- inputs: replicas draw per-rank problems; a head split cuts the one problem ----
    split = args.split
    (h0, h1), seed_off = rank_problem(split, world, rank)
    Hl = h1 - h0
    c = workloads.single_case(T_PROMPT, seed=2 + seed_off, device=dev, ckpt_stride=CKPT)
    dc = workloads.decode_case(N=DEC_N, H=H, D=D, steps=1, seed=4 + seed_off, device=dev)
    if Hl != H:
        c, dc = workloads.head_slice(c, h0, h1), workloads.head_slice(dc, h0, h1)
    cu_dev = c.cu_seqlens.to(dev)
    out = torch.empty(T_PROMPT, Hl, D, device=dev, dtype=torch.bfloat16)
    fin = torch.empty(1, Hl, D, D, device=dev, dtype=torch.float32)
    n_ck = kda.kda_ckpt_count(c.cu_seqlens, CKPT)
    ck = torch.empty(n_ck, Hl, D, D, device=dev, dtype=torch.float32)
    dstate = dc.state
    ds = dc.steps[0]
    dout = torch.empty(DEC_N, Hl, D, device=dev, dtype=torch.bfloat16)
    seg = kda.segments_for(Hl) if args.segments == "auto" else int(args.segments)

    def prefill_call(q, k, v, la, beta, s0, o, f, cp):
        if seg > 0:
            kda.kda_chunk_prefill_segmented(q, k, v, la, beta, s0, T_PROMPT, Hl, D, D, o, kda.KDA_OUT_BF16, f, cp,
                                            CKPT, kda.KDA_DECAY_CHANNEL, 0, seg, stream=stream)
        else:
            kda.kda_chunk_prefill(q, k, v, la, beta, s0, cu_dev, c.cu_seqlens, 1, T_PROMPT, Hl, D, D, o,
                                  kda.KDA_OUT_BF16, f, cp, CKPT, stream)

    def prefill():
        prefill_call(c.q, c.k, c.v, c.log_alpha, c.beta, c.init_state, out, fin, ck)

    def decode():
        kda.kda_decode_step(ds["q"], ds["k"], ds["v"], ds["log_alpha"], ds["beta"], dstate, dout,
                            kda.KDA_OUT_BF16, DEC_N, Hl, D, D, stream)

    for _ in range(max(3, args.warmup)):
        prefill(); decode()
    torch.cuda.synchronize()
    if kda.kda_device_status() != 0:
        raise RuntimeError("device status after warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    # (events for every step: the split between the prefill and decode kernels)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark("t_start")
    start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        prefill()
        ev[i][1].record(stream)
        decode()
        ev[i][2].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t_stop")
    clocks = sampler.stop() if sampler else None
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(stop)
    pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[1].elapsed_time(e[2]) for e in ev]
    if kda.kda_device_status() != 0:
        raise RuntimeError("device status after timed region")

    total_ms, pre_sum, dec_sum = reduce_max([total_ms, sum(pre_ms), sum(dec_ms)], device=dev)
    ms_step = total_ms / args.steps
    pre_avg = pre_sum / args.steps
    dec_avg = dec_sum / args.steps

    value = job_rate(T_PROMPT, world, pre_avg, split)
    hbm, bf16, bf16s, peak_src = read_peaks()
    # per-rank (per-GPU) bytes and FLOPs: the roofline is a single GPU's
    pre_bytes = prefill_algorithmic_bytes(T_PROMPT, n_ck, Hl)
    dec_bytes = decode_algorithmic_bytes(DEC_N, Hl)
    pre_gbs = pre_bytes / (pre_avg / 1e3) / 1e9
    dec_gbs = dec_bytes / (dec_avg / 1e3) / 1e9
    useful_tflops = FLOPS_PER_CHUNK * (T_PROMPT / 64) * Hl / (pre_avg / 1e3) / 1e12

    # ---- end to end through host buffers (pinned), copies inside the timed region ----
    e2e = None
    if not args.no_e2e:
        host = {k: torch.empty_like(getattr(c, k), device="cpu").pin_memory()
                for k in ("q", "k", "v", "log_alpha", "beta")}
        for k2, hv in host.items():
            hv.copy_(getattr(c, k2))
        h_s0 = c.init_state.cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_ck = torch.empty(ck.shape, dtype=ck.dtype).pin_memory()
        h_fin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values()) + h_s0.numel() * 4
        d2h = out.numel() * 2 + ck.numel() * 4 + fin.numel() * 4
        n_e2e = max(2, min(args.steps, 6))
        # Steps are pipelined over two device buffer sets: step i + 1's inputs are copied in
        # (split over N_COPY copy streams) while step i computes and step i - 1's results are
        # copied out.  Every step still moves all of its inputs in and all of its results out.
        N_COPY = 2
        bufs = [dict(d_in={k2: torch.empty_like(getattr(c, k2)) for k2 in host}, s0=torch.empty_like(c.init_state),
                     out=torch.empty_like(out), fin=torch.empty_like(fin), ck=torch.empty_like(ck))
                for _ in range(2)]
        s_in = [torch.cuda.Stream(device=dev) for _ in range(N_COPY)]
        s_out = torch.cuda.Stream(device=dev)
        evs = [{k2: torch.cuda.Event() for k2 in [f"in{j}" for j in range(N_COPY)] + ["comp", "out"]}
               for _ in range(2)]

        def e2e_step(i):
            bf, ev = bufs[i % 2], evs[i % 2]
            for j, sj in enumerate(s_in):               # this buffer's inputs are free again
                sj.wait_event(ev["comp"])
                with torch.cuda.stream(sj):
                    for k2, hv in host.items():          # a 1 / N_COPY row slice of every tensor per stream
                        r0 = hv.shape[0] * j // N_COPY
                        r1 = hv.shape[0] * (j + 1) // N_COPY
                        bf["d_in"][k2][r0:r1].copy_(hv[r0:r1], non_blocking=True)
                    if j == 0:
                        bf["s0"].copy_(h_s0, non_blocking=True)
                    ev["in%d" % j].record(sj)
            for j in range(N_COPY):
                stream.wait_event(ev["in%d" % j])
            stream.wait_event(ev["out"])
            d = bf["d_in"]
            prefill_call(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], bf["s0"], bf["out"], bf["fin"], bf["ck"])
            ev["comp"].record(stream)
            s_out.wait_event(ev["comp"])
            with torch.cuda.stream(s_out):
                h_out.copy_(bf["out"], non_blocking=True)
                h_ck.copy_(bf["ck"], non_blocking=True)
                h_fin.copy_(bf["fin"], non_blocking=True)
                ev["out"].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for sj in (*s_in, s_out):
            sj.wait_event(a)
        for i in range(n_e2e):
            e2e_step(i)
        stream.wait_event(evs[(n_e2e - 1) % 2]["out"])
        b.record(stream)
        torch.cuda.synchronize()
        (e_ms,) = reduce_max([a.elapsed_time(b) / n_e2e], device=dev)
        # the host link itself: one pinned host -> device copy of the largest input, best of 3;
        # the step cannot beat its input bytes at this rate
        hq, dq = host["log_alpha"], bufs[0]["d_in"]["log_alpha"]
        link_ms = []
        for _ in range(3):
            a.record(stream)
            with torch.cuda.stream(stream):
                dq.copy_(hq, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            link_ms.append(a.elapsed_time(b))
        h2d_gbs = hq.numel() * hq.element_size() / (min(link_ms) / 1e3) / 1e9
        floor_ms = h2d / (h2d_gbs * 1e9) * 1e3
        e2e = {"value": job_rate(T_PROMPT, world, e_ms, split), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms, "steps": n_e2e,
               "link": {"h2d_gbs": round(h2d_gbs, 1), "h2d_floor_ms": round(floor_ms, 2),
                        "frac_of_floor": round(floor_ms / e_ms, 3)},
               "note": "prefill only; pinned host inputs copied in, output + checkpoints + final state copied out; "
                       "steps pipelined over two device buffer sets (copy-in of step i+1, split over 2 copy "
                       "streams, and copy-out of step i-1 overlap the prefill of step i)"}
        del host, bufs, h_out, h_ck

    module = None if args.no_module else time_module_path(dev, stream, (h0, h1), seed_off)
    other = None if args.no_other else time_other_rows(dev, stream, (h0, h1), seed_off)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = time_oracle()
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
        cpu["decode_gbs"] = cb["decode_gbs"]

    if rank == 0:
        traffic = read_traffic("kda_prefill_kernel")
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak" if split == "replicas" else "strong", "vs_baseline": None,
            "dtype": "fp16/tf32 MMA, fp32 accumulate + state (bf16 in/out)", "data": "synthetic",
            "config": bench_config(world, split), "heads_per_rank": Hl, "segments": seg,
            "prefill_ms": pre_avg, "decode_ms": dec_avg,
            "decode": {"value": dec_gbs * world, "unit": "GB/s", "tokens_per_s": job_rate(DEC_N, world, dec_avg, split),
                       "frac_of_hbm_peak": dec_gbs / hbm},
            "roofline": {"bound": "hbm", "achieved": pre_gbs, "peak": hbm, "unit": "GB/s",
                         "frac": pre_gbs / hbm, "traffic": traffic, "kernel": "kda_prefill_kernel",
                         "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_launch": pre_bytes},
            "useful_flops": {"tflops": useful_tflops, "frac_of_bf16_peak": useful_tflops / bf16,
                             "frac_of_bf16_sustained": useful_tflops / bf16s, "peak_source": peak_src},
            "kv_throughput": {"value": kv_state_bytes(n_ck, Hl) * world / (pre_avg * 1e-3) / 1e9, "unit": "GB/s",
                              "state_bytes_per_prefill": kv_state_bytes(n_ck, Hl),
                              "note": "final state + checkpoints written per prefill / prefill time"},
            "clocks": clocks, "e2e": e2e, "gpu_launches": (2 if seg == 0 else 6) * args.steps, "cpu_baseline": cpu,
            "module": module, "other": other,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
