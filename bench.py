"""Batch-1 greedy decode throughput of the 2B fp16 Llama-style workload on GB300, as one JSON line.

A step is one kie_decode of 1,024 tokens after a 128-token prompt (prefill untimed for `value`): one launch
of the persistent monokernel. `value` = decode tokens / device time (CUDA events on the library's stream);
`e2e` = the same tokens through the public host-buffer API (reset + prefill from a host prompt + decode
into a host array, wall clock), so it includes the prompt and both copies. Weights (3.9 GB) are larger than
L2 and every token streams them all, so no L2 flush is needed between steps.

--impl reference times the CPU oracle (oracle/, plain C) on the host cores on a bounded sample of the same
workload. With N > 1 (torchrun) every rank runs an independent replica: the path has no data exchange.

Other modes (not the headline line): --long runs the long-context workload (prompt 8,192, 512 new tokens);
--moe the sparse-MoE workload (24 layers, 64 FP8 experts of width 1,024, top 4; prompt 256, 512 new tokens),
whose MBU counts the bytes a token actually streams (attention, router, the 4 routed experts, LM head);
--prefill N times the batched prefill of an N-token prompt (tensor-core projections, split causal attention);
--gemv-sweep prints one JSON line per standalone GEMV shape (GB/s, cold HBM); --phase-gemv does the same for
the decode's five projection shapes of the 2B model (the phase-split view of the weight stream).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 decode tok/s, 2B fp16 on 1 GB300; MBU vs HBM peak"
WORKLOAD = "llama2b_p128_n1024"
PROMPT, NEW = 128, 1024
MOE_METRIC = "batch-1 decode tok/s, sparse MoE (64 FP8 experts, top 4) on 1 GB300; MBU over active bytes"


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def phase_bytes(model, c):
    """Algorithmic bytes of each phase of one layer (and of the LM head) at c attended positions."""
    d, dh, F = model.d_model, model.head_dim, model.ffn_dim
    out = {"qkv": 2 * (model.n_heads + 2 * model.n_kv_heads) * dh * d, "att": 2 * 2 * model.n_kv_heads * dh * c,
           "wo": 2 * d * model.n_heads * dh, "gu": 2 * 2 * F * d, "down": 2 * d * F, "lm": 2 * model.vocab * d}
    if getattr(model, "n_experts", 0):
        k = model.top_k
        out.update(router=2 * model.n_experts * d, egu=k * (2 * F * d + 4 * 2 * F), edown=k * (d * F + 4 * d))
    return out


def phase_names(model):
    """The grid phases of one layer, in order (sparse MoE: the router is folded into the QKV and WO phases, and the
    expert gate/up phase starts with the selection)."""
    if getattr(model, "n_experts", 0):
        return ["qkv", "att", "wo", "egu", "edown"]
    return ["qkv", "att", "wo", "gu", "down"]


def phase_breakdown(dec, model, prompt_len, new):
    """Per-phase time from the grid-barrier trace of the last launch (the first tokens it recorded): a phase
    runs from the earliest departure from the previous barrier to the last arrival at its own; the release
    latency is the gap between the last arrival at a barrier and the earliest departure from it."""
    import numpy as np
    names = phase_names(model)
    per_tok = len(names) * model.n_layers + 1
    toks = min(new, 4096 // per_tok)
    if toks < 2:
        return None
    arrive, wait = dec.barrier_trace(0, toks * per_tok)
    arrive = arrive.astype(np.float64)
    leave = arrive + wait
    per = {n: [] for n in names + ["lm"]}
    release = []
    for k in range(1, arrive.shape[0]):
        j = k % per_tok
        name = "lm" if j == per_tok - 1 else names[j % len(names)]
        per[name].append((arrive[k].max() - leave[k - 1].min()) / 1e3)
        release.append((leave[k].min() - arrive[k].max()) / 1e3)
    c_mid = prompt_len + 1 + toks // 2
    b = phase_bytes(model, c_mid)
    stamps = np.unique(arrive)
    step = float(np.min(np.diff(stamps))) if stamps.size > 1 else 0.0
    out = {"tokens": f"{toks} tokens from c = {prompt_len + 1}", "timer_step_ns": step,
           "note": "%globaltimer stamps advance in timer_step_ns steps: a single phase time is quantised to it; "
                   "us is the mean over the recorded phases, median_us the (quantised) median",
           "release_latency_us": float(np.mean(release)),
           "barrier_us_per_token": float(np.mean(release)) * per_tok}
    for n, v in per.items():
        us = float(np.mean(v))  # the mean over many phases is finer than one timer step
        out[n] = {"us": us, "gbs": b[n] / us / 1e3, "median_us": float(np.median(v))}
    return out


def gemv_sweep(args, shapes=None, label="standalone fp16 GEMV GB/s (one launch each, cold HBM, CUDA graph)"):
    """y = W x for the 25 sweep shapes (or `shapes`) through kie_gemv. The launches are captured in a CUDA graph (so the
    host-side cost of each call is not timed) that cycles over enough packed copies of W that every launch
    reads cold HBM (at least 4x L2 of distinct bytes); time per launch = replay time / launches."""
    import torch

    import persistent_monokernel_decode_gb300 as kie
    import synth
    from synth.configs import GEMV_SHAPES
    kie.build()
    shapes = shapes or GEMV_SHAPES
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    peaks, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    for sh in shapes:
        W, x = synth.gemv_operands(sh)
        Wd = torch.from_numpy(W.view("int16")).cuda()
        xd = torch.from_numpy(x.view("int16")).cuda()
        copies = max(1, -(-4 * l2 // (2 * sh.M * sh.K)))
        packed = [kie.gemv_pack(Wd) for _ in range(copies)]
        y = torch.empty(sh.M, dtype=torch.float32, device="cuda")
        per_graph = max(copies, 16)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                kie.gemv(packed[i % copies], xd, sh.M, sh.K, y=y)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for i in range(per_graph):
                    kie.gemv(packed[i % copies], xd, sh.M, sh.K, y=y)
            g.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / (args.steps * per_graph)
        gbs = sh.bytes() / t / 1e9
        print(json.dumps({"metric": label, "phase": getattr(sh, "phase", None), "M": sh.M, "K": sh.K, "value": gbs, "unit": "GB/s", "us": t * 1e6, "copies": copies,
                          "frac_of_peak": gbs / peaks["hbm_gbs"], "peak_kind": peak_kind}), flush=True)
        del g, packed, Wd, xd, y


def phase_shapes():
    """The decode's projections of the 2B model as standalone GEMV shapes (seeded like the sweep)."""
    import dataclasses

    from synth.configs import TWO_B, GemvShape

    @dataclasses.dataclass(frozen=True)
    class PhaseShape(GemvShape):
        phase: str = ""

    m = TWO_B
    d, dq, F = m.d_model, m.n_heads * m.head_dim, m.ffn_dim
    dims = [("qkv", (m.n_heads + 2 * m.n_kv_heads) * m.head_dim, d), ("wo", d, dq), ("gate_up", 2 * F, d),
            ("down", d, F), ("lm_head", m.vocab, d)]
    return [PhaseShape(M, K, 2000 + i, phase=name) for i, (name, M, K) in enumerate(dims)]


def profiled_traffic(workload, digest):
    """DRAM bytes per decode launch from the committed ncu summary of this workload, if that capture was taken
    from the same kernel sources (the summary's `source_digest` line); otherwise None."""
    import re
    path = os.path.join(ROOT, "profiles", f"decode_kernel_{workload}_dram.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"^source_digest:\s*([0-9a-f]+)\s*$", text, re.M)
    t = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)\s*$", text, re.M)
    if not m or not t or m.group(1) != digest:
        return None
    return float(t.group(1))


def roofline(bytes_per_step, step_s, peak_gbs):
    """Achieved GB/s of a step that must move bytes_per_step in step_s seconds, and its fraction of peak_gbs
    (MBU when the bytes are the weight and K/V bytes the tokens read)."""
    achieved = bytes_per_step / step_s / 1e9
    return achieved, achieved / peak_gbs


def algorithmic_bytes(model, prompt_len, n):
    """Bytes one decode of n tokens must move: every weight once per token, plus the K/V prefix it attends
    over (the token at position p attends over p + 1 positions)."""
    w = model.weight_bytes_per_token() * n
    kv = sum(model.kv_bytes_per_token(prompt_len + t + 1) for t in range(n))
    return w + kv


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc = index, None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x, pg, device="cuda"):
    """The largest x over all ranks of the process group (x itself without one): the job's time is the
    slowest rank's."""
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], device=device, dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_rank, step_s):
    """Whole-job tokens/s of `world` independent replicas that each decode tokens_per_rank in step_s (the
    slowest rank's step time)."""
    return world * tokens_per_rank / step_s


def emit(line, rank):
    """The JSON line is printed by rank 0 only."""
    if rank == 0:
        print(json.dumps(line), flush=True)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, world, rank):
    """The CPU oracle, timed on this host's cores (rank 0 only)."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    import synth
    from synth.configs import TWO_B

    per_step = 2  # decode forwards per step: a bounded sample (~1-3 s of CPU time each on 16 cores)
    w = synth.model_weights(TWO_B)
    prompt = synth.tokens(TWO_B.seed, PROMPT, TWO_B.vocab)
    m = oracle.Model(TWO_B, w, PROMPT + (args.warmup + args.steps) * per_step + 1, 32)
    ctx_prompt = prompt[:8]  # short untimed prefill: the sample measures decode forwards only
    cur = m.prefill(ctx_prompt)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for _ in range(per_step):
            cur = m.forward(oracle.argmax(cur))
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = args.steps * per_step / total
    cores = oracle.threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{per_step} greedy decode forwards per step after an "
                   f"8-token prefill (2B model, full weights)", "weights": "fp16", "kv_cache": "fp16"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} x {per_step} decode forwards of the 2B model"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_sample(seconds_budget=15.0, max_forwards=400, model=None, weights=None):
    """The oracle as it stands on the host cores: greedy decode forwards of the 2B model (or `model` with
    `weights`), for about seconds_budget of CPU time (at most max_forwards)."""
    import oracle
    import synth
    from synth.configs import TWO_B

    if model is None:
        model, weights = TWO_B, synth.model_weights(TWO_B)
    prompt = synth.tokens(model.seed, 8, model.vocab)
    m = oracle.Model(model, weights, len(prompt) + max_forwards + 1, 32)
    cur = m.prefill(prompt)
    n, t0 = 0, time.perf_counter()
    while n < max_forwards:
        cur = m.forward(oracle.argmax(cur))
        n += 1
        if time.perf_counter() - t0 > seconds_budget:
            break
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tok/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{n} greedy decode forwards of the {model.name} model after an 8-token prefill ({dt:.1f} s)"}


def prefill_bench(args):
    """kie_prefill of an N-token prompt (reset + prefill, CUDA events on the library's stream): tokens/s and the
    projections' useful TFLOP/s (2 x parameters x tokens; the attention's FLOP are reported separately)."""
    import dataclasses

    import torch

    import persistent_monokernel_decode_gb300 as kie
    import synth
    from synth.configs import TWO_B

    n = args.prefill
    model = TWO_B if args.layers == TWO_B.n_layers else dataclasses.replace(TWO_B, n_layers=args.layers)
    kie.build()
    w = synth.model_weights(model)
    prompt = synth.tokens(model.seed, n, model.vocab)
    dec = kie.Decoder(model, w, max_seq=n + 16)
    del w
    times = []
    for i in range(args.warmup + args.steps):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(dec.stream)
        dec.reset()
        dec.prefill(prompt)
        e1.record(dec.stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
    dec.close()
    t = sum(times) / len(times)
    d, dh, F = model.d_model, model.head_dim, model.ffn_dim
    params = model.n_layers * ((model.n_heads + 2 * model.n_kv_heads) * dh * d + d * model.n_heads * dh + 3 * F * d)
    att = 4 * model.n_heads * dh * sum(range(1, n + 1)) * model.n_layers
    print(json.dumps({"metric": "batched prefill tok/s", "value": n / t, "unit": "tok/s", "ms": 1e3 * t,
                      "steps": args.steps, "warmup": args.warmup, "tokens": n, "layers": model.n_layers,
                      "projection_tflops_useful": 2 * params * n / t / 1e12, "attention_gflop": att / 1e9}),
          flush=True)


def attention_phase(args):
    """The decode's split-KV attention step alone (kie_profile_attention: the same device function and grid
    barrier), on the 2B model with its cache filled to c positions: the step's time per layer from the kernel's
    own clock (first CTA start to end, 25 layers per launch, so the launch itself is not in it; median over
    --steps launches) and the K/V bytes it must read (2 x Hkv x dh x c fp16 per layer), one JSON line per c."""
    import dataclasses

    import torch

    import persistent_monokernel_decode_gb300 as kie
    import synth
    from synth.configs import TWO_B
    kie.build()
    model = TWO_B if args.layers == TWO_B.n_layers else dataclasses.replace(TWO_B, n_layers=args.layers)
    layers = model.n_layers
    w = synth.model_weights(model)
    peaks, peak_kind = measured_peaks()
    cs = tuple(int(v) for v in args.contexts.split(","))
    dec = kie.Decoder(model, w, max_seq=max(cs) + 8)
    del w
    for c in cs:
        dec.reset()
        dec.prefill(synth.tokens(model.seed, c, model.vocab))
        times = []
        for i in range(args.warmup + args.steps):
            dec.profile_attention(c, layers)
            torch.cuda.synchronize()
            if i >= args.warmup:
                times.append(dec.barrier_stats()["total_ns"] * 1e-9)
        t_layer = statistics.median(times) / layers
        kv = 2 * 2 * model.n_kv_heads * model.head_dim * c
        print(json.dumps({"metric": "split-KV attention step alone, per layer", "c": c, "layers": layers,
                          "us_per_layer": t_layer * 1e6,
                          "kv_bytes_per_layer": kv, "GBs": kv / t_layer / 1e9,
                          "frac_of_peak": kv / t_layer / 1e9 / peaks["hbm_gbs"], "peak_kind": peak_kind,
                          "timing": f"kernel clock over {layers} layers per launch, one grid barrier per layer",
                          "steps": args.steps, "warmup": args.warmup}), flush=True)
    dec.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kie", choices=["kie", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=25, help="fewer layers of the same widths (profiling cases)")
    ap.add_argument("--prompt", type=int, default=PROMPT)
    ap.add_argument("--decode", type=int, default=NEW)
    ap.add_argument("--long", action="store_true", help="the long-context workload: prompt 8,192, 512 new tokens")
    ap.add_argument("--prefill", type=int, default=0, metavar="N",
                    help="time the batched prefill of an N-token prompt of the 2B model (or --layers of its widths)")
    ap.add_argument("--moe", action="store_true",
                    help="the sparse-MoE workload (64 FP8 experts, top 4): prompt 256, 512 new tokens")
    ap.add_argument("--gemv-sweep", action="store_true", help="standalone GEMV GB/s for the 25 sweep shapes")
    ap.add_argument("--contexts", default="129,145,300,600,1152,8192",
                    help="attended positions for --phase-attention, comma-separated")
    ap.add_argument("--phase-attention", action="store_true",
                    help="the decode's split-KV attention step alone, 2B model, c from 129 to 8,192")
    ap.add_argument("--phase-gemv", action="store_true",
                    help="the decode's five projection shapes of the 2B model through the standalone GEMV (GB/s each)")
    args = ap.parse_args()
    if args.long:
        args.prompt, args.decode = 8192, 512
    if args.moe:
        args.prompt = 256 if args.prompt == PROMPT else args.prompt
        args.decode = 512 if args.decode == NEW else args.decode
    if args.gemv_sweep:
        gemv_sweep(args)
        return
    if args.phase_attention:
        attention_phase(args)
        return
    if args.phase_gemv:
        gemv_sweep(args, phase_shapes(), "2B decode projection as one standalone GEMV: GB/s (cold HBM, CUDA graph)")
        return
    world, rank, local = dist_setup()
    if args.prefill:
        prefill_bench(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import dataclasses

    import numpy as np
    import torch

    import persistent_monokernel_decode_gb300 as kie
    import synth
    from synth.configs import MOE_M, TWO_B

    prompt_len, new = args.prompt, args.decode
    if args.moe:
        layers = MOE_M.n_layers if args.layers == 25 else args.layers
        model = MOE_M if layers == MOE_M.n_layers else dataclasses.replace(MOE_M, n_layers=layers)
        workload = "moe_p256_n512" if (layers, prompt_len, new) == (24, 256, 512) else \
            f"moe_L{layers}_p{prompt_len}_n{new}"
    else:
        model = TWO_B if args.layers == TWO_B.n_layers else dataclasses.replace(TWO_B, n_layers=args.layers)
        workload = WORKLOAD if (args.layers, prompt_len, new) == (25, PROMPT, NEW) else \
            ("llama2b_p8192_n512" if (args.layers, prompt_len, new) == (25, 8192, 512) else
             f"llama2b_L{args.layers}_p{prompt_len}_n{new}")

    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    kie.build()

    w = synth.moe_weights(model) if args.moe else synth.model_weights(model)
    prompt = synth.tokens(model.seed, prompt_len, model.vocab)
    dec = kie.Decoder(model, w, max_seq=prompt_len + new)
    if not args.moe:
        del w
    out = torch.empty(new, dtype=torch.int32, device="cuda")
    stream = dec.stream

    def prefill():
        dec.reset()
        dec.prefill(prompt)

    for _ in range(args.warmup):
        prefill()
        dec.decode_async(new, out)
        dec.sync()

    clocks = ClockSampler(local)
    times = []
    stats = None
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for _ in range(args.steps):
        prefill()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dec.decode_async(new, out)
        e1.record(stream)
        dec.sync()
        times.append(e0.elapsed_time(e1) / 1e3)
    torch.cuda.synchronize()
    clk = clocks.stop()
    stats = dec.barrier_stats()
    phases = phase_breakdown(dec, model, prompt_len, new)
    step_s = max_over_ranks(statistics.median(times), pg)
    value = replica_throughput(world, new, step_s)

    # end to end through the host-buffer API: reset + prefill(host prompt) + decode(n, host tokens)
    e2e_times = []
    host_out = np.empty(new, dtype=np.int32)
    for i in range(args.warmup + args.steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dec.reset()
        dec.prefill(prompt)
        host_out[:] = dec.decode(new)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            e2e_times.append(dt)
    e2e_step = max_over_ranks(statistics.median(e2e_times), pg)

    peaks, peak_kind = measured_peaks()
    bytes_launch = algorithmic_bytes(model, prompt_len, new)
    achieved, frac = roofline(bytes_launch, step_s, peaks["hbm_gbs"])
    line = {
        "metric": MOE_METRIC if args.moe else METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload, "prompt": prompt_len, "decode_tokens": new,
                   "weights": "fp16 attention/router/LM head, FP8 E4M3 experts" if args.moe else "fp16",
                   "kv_cache": "fp16",
                   "l2": (f"no flush: {model.weight_bytes_per_token() / 1e9:.2f} GB of weights (> 129 MB L2) "
                          "streamed per token"),
                   "parallelism": "replicas" if world > 1 else "single GPU", "n_cta": dec.n_cta},
        "e2e": {"value": replica_throughput(world, new, e2e_step), "unit": "tok/s", "h2d_bytes_per_step": prompt_len * 4,
                "d2h_bytes_per_step": new * 4 + 8,
                "timed": f"reset + prefill({prompt_len}-token host prompt) + decode({new} -> host array), wall clock"},
        "statistic": f"median over the {args.steps} timed launches (CUDA events on the library's stream), "
                     "max over ranks",
        "step_ms_all": [round(1e3 * t, 4) for t in times],
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": frac, "traffic": profiled_traffic(workload, kie.source_digest()),
                     "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "algorithmic_bytes_per_launch": bytes_launch},
        "mbu": {"measured_peak": achieved / peaks["hbm_gbs"], "spec_8tbs": achieved / 8000.0},
        "barriers": {"per_token": stats["barriers"] / new, "mean_latency_ns": stats["mean_latency_ns"],
                     "mean_wait_ns": stats["mean_wait_ns"],
                     "wait_us_per_token": stats["mean_wait_ns"] * stats["barriers"] / new / 1e3},
        "phases": phases,
        "clocks": clk,
    }
    dec.close()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(model=model, weights=w) if args.moe else cpu_baseline_sample()
    emit(line, rank)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
