"""Run one KDA workload a few times through the C ABI (for profilers and quick timing).

  python -m kimi_delta_attention_06_gb300.run_case --what prefill --T 8192 [--H 32] [--D 128] [--reps 2]
  python -m kimi_delta_attention_06_gb300.run_case --what varlen [--H 32] [--D 128] [--reps 2]
      (prefill / varlen also take --decay channel|head|none: KDA, Gated DeltaNet, DeltaNet;
       prefill / varlen --segments P run kda_chunk_prefill_segmented(_ex) with P segments)
  python -m kimi_delta_attention_06_gb300.run_case --what decode --N 512 [--H 32] [--D 128] [--reps 2]
  python -m kimi_delta_attention_06_gb300.run_case --what decode_multi --N 512 --K 4 [--commit 1] [--reps 2]
  python -m kimi_delta_attention_06_gb300.run_case --what prep --T 145408 [--reps 2]     (input preparation)
  python -m kimi_delta_attention_06_gb300.run_case --what outnorm --T 145408 [--reps 2]  (output norm)

Inputs are the seeded synthetic tensors of workloads.py, generated on the GPU
(varlen: 16 packed sequences of log-uniform length, about 280k tokens).
Prints the CUDA-event time of each repetition and the median rate of the
repetitions after the first.
"""
from __future__ import annotations

import argparse

import torch

from . import build, kda, workloads


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--what", choices=["prefill", "varlen", "decode", "decode_multi", "prep", "outnorm"],
                    default="prefill")
    ap.add_argument("--K", type=int, default=4, help="tokens per sequence (decode_multi)")
    ap.add_argument("--commit", type=int, default=0, help="decode_multi: 1 writes the states back")
    ap.add_argument("--decay", choices=["channel", "head", "none"], default="channel",
                    help="prefill decay layout (per channel = KDA, per head = Gated DeltaNet, none = DeltaNet)")
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--N", type=int, default=512)
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--ckpt", type=int, default=32768)
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--segments", type=int, default=0, help="prefill: segments of kda_chunk_prefill_segmented")
    a = ap.parse_args(argv)
    build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    if a.what in ("prefill", "varlen"):
        if a.what == "prefill":
            c = workloads.single_case(a.T, seed=2, device=dev, H=a.H, D=a.D, ckpt_stride=a.ckpt)
        else:
            c = workloads.varlen_case(device=dev, H=a.H, D=a.D, ckpt_stride=a.ckpt)
        T, N = c.T, c.N
        cu = c.cu_seqlens.to(dev)
        decay = {"channel": kda.KDA_DECAY_CHANNEL, "head": kda.KDA_DECAY_HEAD, "none": kda.KDA_DECAY_NONE}[a.decay]
        la = {kda.KDA_DECAY_CHANNEL: c.log_alpha, kda.KDA_DECAY_HEAD: c.log_alpha[:, :, 0].contiguous(),
              kda.KDA_DECAY_NONE: None}[decay]
        out = torch.empty(T, a.H, a.D, device=dev, dtype=torch.bfloat16)
        fin = torch.empty(N, a.H, a.D, a.D, device=dev)
        nck = kda.kda_ckpt_count(c.cu_seqlens, a.ckpt)
        ck = torch.empty(max(nck, 1), a.H, a.D, a.D, device=dev)

        def run():
            if a.segments > 0 and a.what == "varlen":
                kda.kda_chunk_prefill_segmented_ex(c.q, c.k, c.v, la, c.beta, c.init_state, c.cu_seqlens, N, T, a.H,
                                                   a.D, a.D, out, kda.KDA_OUT_BF16, fin, ck if nck else None, a.ckpt,
                                                   decay, None, a.segments, stream=stream)
            elif a.segments > 0 and a.what == "prefill":
                kda.kda_chunk_prefill_segmented(c.q, c.k, c.v, la, c.beta, c.init_state, T, a.H, a.D, a.D, out,
                                                kda.KDA_OUT_BF16, fin, ck if nck else None, a.ckpt, decay, 0,
                                                a.segments, stream=stream)
            else:
                kda.kda_chunk_prefill_ex(c.q, c.k, c.v, la, c.beta, c.init_state, cu, c.cu_seqlens, N, T, a.H,
                                         a.D, a.D, out, kda.KDA_OUT_BF16, fin, ck if nck else None, a.ckpt, decay,
                                         stream=stream)
        units, count = f"{T} tokens, {N} sequences, decay {a.decay}, segments {a.segments}", T
    elif a.what in ("prep", "outnorm"):
        g = torch.Generator(device=dev).manual_seed(6)
        T, H, D = a.T, a.H, a.D
        cu_host = torch.tensor([0, T], dtype=torch.int32)
        cu = cu_host.to(dev)
        if a.what == "prep":
            xs = [torch.randn(T, H, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(3)]
            w = torch.randn(3, H, D, 4, generator=g, device=dev) * 0.5
            ar = torch.randn(T, H, D, generator=g, device=dev) - 2.0
            br = torch.randn(T, H, generator=g, device=dev).to(torch.bfloat16)
            outs = [torch.empty(T, H, D, device=dev, dtype=torch.bfloat16) for _ in range(3)]
            la = torch.empty(T, H, D, device=dev)
            be = torch.empty(T, H, device=dev, dtype=torch.bfloat16)

            def run():
                kda.kda_prepare_inputs(xs[0], xs[1], xs[2], w, None, ar, br, cu, cu_host, 1, T, H, D, 1,
                                       outs[0], outs[1], outs[2], la, be, stream)
            nbytes = T * H * (3 * 2 * D + 4 * D + 2) * 2          # read and write the same bytes
        else:
            o = torch.randn(T, H, D, generator=g, device=dev).to(torch.bfloat16)
            gam = torch.rand(H, D, generator=g, device=dev) + 0.5
            y = torch.empty_like(o)

            def run():
                kda.kda_output_norm(o, kda.KDA_OUT_BF16, gam, 1e-6, y, T, H, D, stream)
            nbytes = T * H * D * 2 * 2
        units, count = f"{T} tokens x {H} heads ({nbytes / 1e9:.3f} GB moved)", T
    elif a.what == "decode_multi":
        d = workloads.decode_case(N=a.N, H=a.H, D=a.D, steps=a.K, seed=4, device=dev)
        tok = {key: torch.stack([s[key] for s in d.steps], dim=1).contiguous()
               for key in ("q", "k", "v", "log_alpha", "beta")}
        out = torch.empty(a.N, a.K, a.H, a.D, device=dev, dtype=torch.bfloat16)

        def run():
            kda.kda_decode_multi(tok["q"], tok["k"], tok["v"], tok["log_alpha"], tok["beta"], d.state, a.N, None,
                                 None, a.commit, out, kda.KDA_OUT_BF16, a.N, a.K, a.H, a.D, a.D, stream=stream)
        units, count = f"{a.N} sequences x {a.K} tokens, commit={a.commit}", a.N * a.K
    else:
        d = workloads.decode_case(N=a.N, H=a.H, D=a.D, steps=1, seed=4, device=dev)
        s = d.steps[0]
        out = torch.empty(a.N, a.H, a.D, device=dev, dtype=torch.bfloat16)

        def run():
            kda.kda_decode_step(s["q"], s["k"], s["v"], s["log_alpha"], s["beta"], d.state, out,
                                kda.KDA_OUT_BF16, a.N, a.H, a.D, a.D, stream)
        units, count = f"{a.N} sequences", a.N
    times = []
    for i in range(a.reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
        print(f"{a.what} rep {i}: {times[-1]:.3f} ms ({units})")
    if len(times) > 1:
        med = sorted(times[1:])[(len(times) - 1) // 2]
        print(f"{a.what} median of reps 1..{len(times) - 1}: {med:.3f} ms = {count / med * 1e3:.4g} "
              f"{'sequences' if a.what == 'decode' else 'tokens'}/s")
    st = kda.kda_device_status()
    if st != 0:
        raise SystemExit(f"device status {st}")


if __name__ == "__main__":
    main()
