#!/usr/bin/env python3
"""Benchmark: KDA forward + backward tokens/s on the packed 4-document batch
(T = 261392, H = 16, D = 128) on one GB300, with the roofline fraction of the
dominant kernel, end-to-end throughput through the C ABI with host buffers,
and the FP64 oracle timed on the host cores as a CPU baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdr|reference]

One step = one forward (saving for the backward) + one backward over the whole
batch, inputs resident in HBM.  Between timed steps a 256 MiB buffer is written
to flush L2 (the inputs themselves are larger than L2).  Under torchrun each
rank runs its own replica of the batch (weak scaling; no collective on the data
path); the slowest rank's time counts.  Rank 0 prints one JSON line.

--impl reference times the FP64 CPU oracle (the only reference there is) on a
bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA fwd+bwd tokens/s (T=261392, H=16, D=128, 1 GB300); % of roofline"
UNIT = "tokens/s"

# Algorithmic bytes and FLOPs per (token, value head) of each kernel: every
# input read once and every output written once at its stored precision
# (BF16 I/O, FP32 gates and intermediates), and the chunk-64 matrix products
# counted at 2 flops per multiply-add (triangular 64x64 factors at half).
C, D = 64, 128
_TILE = D * 4           # one FP32 row of a [64][128] intermediate
_STATE = D * D * 4 / C  # one FP32 128x128 state per chunk, per token
KERNEL_MODEL = {
    # name: (bytes per token-head, flops per token-head)
    "prep": (3 * 2 * D + 4 * D + 2 + 4 * _TILE + 3 * C * 4 + 4 * D / C,
             2 * (2 * 0.5 * C * D) + 2 * (2 * 0.5 * C * D) + C * C / 3),
    # state walk with the outputs: reads w, u, Kd^T, Q Gamma, Aqk, gamma; writes
    # Delta, the BF16 state tape and the BF16 output.
    "walk_fwd": (4 * _TILE + C * 4 + 4 * D / C + _TILE + _STATE / 2 + 2 * D,
                 3 * (2 * D * D) + 2 * 0.5 * C * D),
    "walk_bwd": (C * 4 + 3 * _TILE + 2 * D + _STATE / 2 + _TILE, 2 * (2 * D * D) + 2 * D * D + 2 * 0.5 * C * D),
    "grad_state": (2 * D + _STATE + 2 * _TILE + 3 * _TILE + 4 * D / C + C * 4, 3 * (2 * D * D)),
    "grad": (3 * 2 * D + 4 * D + 2 + 2 * D + 3 * _TILE + 3 * C * 4 + 2 * _TILE + 3 * _TILE + 3 * 2 * D + 4 * D + 2,
             11 * (2 * 0.5 * C * D) + 2 * (2 * C * D)),
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("gdr", "reference"), default="gdr")
    ap.add_argument("--workload", default="kda_pack_h16")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ckpt", action="store_true")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks, power and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.2)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, pw, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                    pw.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(sm)}


def source_hash():
    """Hash of the sources that define the measured kernels (the C-ABI file,
    which holds only planning and validation, is left out)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_varlen_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name == "gdr_api.cu":
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes per (token, value head) of `kernel` from the committed ncu
    summary, if it was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    rec = data.get(kernel)
    if not rec or rec.get("source_hash") != source_hash():
        return None
    return rec.get("dram_bytes_per_token_head")


def oracle_sample(wl, x_host, max_tokens: int):
    """Run the FP64 oracle fwd+bwd on the first `max_tokens` tokens of every
    document, all heads; returns (token-heads processed, seconds, threads)."""
    import oracle
    cu = wl.cu_seqlens
    idx, lens = [], []
    for n in range(len(wl.lengths)):
        s = cu[n]
        m = min(max_tokens, wl.lengths[n])
        idx.extend(range(s, s + m))
        lens.append(m)
    import torch
    sel = torch.tensor(idx, dtype=torch.long)
    f = {k: v.index_select(0, sel).double().numpy() for k, v in x_host.items()}
    cu_s = [0]
    for m in lens:
        cu_s.append(cu_s[-1] + m)
    threads = oracle.hardware_threads()
    t0 = time.perf_counter()
    oracle.run(f["q"], f["k"], f["v"], f["g"], f["beta"], cu_s, D ** -0.5, dout=f["dout"], threads=threads)
    dt = time.perf_counter() - t0
    return sum(lens) * wl.HV, dt, threads


def run_reference(args):
    import synth
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = synth.workload(args.workload)
    x = synth.make_inputs(wl.variant, wl.T, wl.Hqk, wl.HV, D, seed=0, device="cpu")
    sample_tokens = 1024
    for _ in range(args.warmup):
        oracle_sample(wl, x, 256)
    th, secs = 0, 0.0
    for _ in range(args.steps):
        n, dt, threads = oracle_sample(wl, x, sample_tokens)
        th += n
        secs += dt
    value = th / secs / wl.HV
    sample = (f"first {sample_tokens} tokens of each of the {len(wl.lengths)} documents, all {wl.HV} heads, "
              f"fwd+bwd, per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.HV, "D": D, "docs": list(wl.lengths)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    import gated_delta_rule_varlen_gb300 as gdr
    import synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    gdr.load()

    wl = synth.workload(args.workload)
    T, Hqk, HV = wl.T, wl.Hqk, wl.HV
    cu_host = wl.cu_seqlens
    x = synth.make_inputs(wl.variant, T, Hqk, HV, D, seed=0, device=dev)
    cu_d = torch.tensor(cu_host, dtype=torch.int32, device=dev)
    scale = D ** -0.5
    kda = wl.variant == "kda"
    fwd = gdr.kda_fwd if kda else gdr.gdn_fwd
    bwd = gdr.kda_bwd if kda else gdr.gdn_bwd
    wsb = gdr.kda_workspace_bytes(T, HV, cu_host) if kda else gdr.gdn_workspace_bytes(T, Hqk, HV, cu_host)
    saved = torch.empty(wsb[0], dtype=torch.uint8, device=dev)
    scratch = torch.empty(max(wsb), dtype=torch.uint8, device=dev)
    out = torch.empty((T, HV, D), dtype=torch.bfloat16, device=dev)
    ht = torch.empty((len(wl.lengths), HV, D, D), dtype=torch.float32, device=dev)
    grads = {"dq": torch.empty_like(x["q"]), "dk": torch.empty_like(x["k"]), "dv": torch.empty_like(x["v"]),
             "dg": torch.empty_like(x["g"]), "dbeta": torch.empty_like(x["beta"])}
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def fwd_call(xx, save=True):
        return fwd(xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_d, cu_host, scale, out=out, ht=ht,
                   saved=saved if save else None, save_for_bwd=save, scratch=None if save else scratch)

    def bwd_call(xx):
        return bwd(xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_d, cu_host, scale, xx["dout"], saved,
                   scratch=scratch, grads=grads)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 1)):
        fwd_call(x)
        bwd_call(x)
    barrier()

    # ---- timed region: K steps of fwd + bwd -------------------------------
    sampler = ClockSampler(local)
    sampler.start()
    gdr.gdr_profile_enable(True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches_before = 0
    barrier()
    wall0 = time.perf_counter()
    for e0, e1, e2 in evs:
        flush.zero_()
        e0.record(stream)
        fwd_call(x)
        e1.record(stream)
        bwd_call(x)
        e2.record(stream)
    barrier()
    wall = time.perf_counter() - wall0
    gdr.gdr_profile_enable(False)
    clocks = sampler.stop()
    kern = gdr.gdr_profile_report()
    t_fwd = [a.elapsed_time(b) for a, b, _ in evs]
    t_bwd = [b.elapsed_time(c) for _, b, c in evs]
    t_step = [f + b for f, b in zip(t_fwd, t_bwd)]
    ms_step = statistics.mean(t_step)
    if world > 1:
        tt = torch.tensor([ms_step], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_step = float(tt.item())
    value = world * T / (ms_step / 1e3)
    gpu_launches = sum(v[0] for v in kern.values())

    # ---- ckpt: forward (no save), forward (save), backward -----------------
    ckpt_ms = None
    if not args.no_ckpt:
        cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(max(args.steps // 4, 2))]
        barrier()
        for a, b in cev:
            flush.zero_()
            a.record(stream)
            fwd_call(x, save=False)
            fwd_call(x, save=True)
            bwd_call(x)
            b.record(stream)
        barrier()
        ckpt_ms = statistics.median([a.elapsed_time(b) for a, b in cev])

    # ---- end to end through the C ABI with host buffers --------------------
    # Every step copies its inputs from pinned host memory and its results
    # (out and every gradient) back.  Steps are pipelined the way a training
    # loop with host-resident data runs them: device inputs and outputs are
    # double-buffered, step s+1's inputs are copied in and step s-1's results
    # copied out on two copy streams while step s computes.  The timed region
    # runs from before the first input copy to after the last result copy.
    e2e = None
    if not args.no_e2e:
        names_in = ("q", "k", "v", "g", "beta", "dout")
        host_in = {k: x[k].cpu().pin_memory() for k in names_in}
        dev_in = [{k: x[k] for k in names_in}, {k: torch.empty_like(x[k]) for k in names_in}]
        dev_out = [{"out": out, **grads}, None]
        dev_out[1] = {k: torch.empty_like(v) for k, v in dev_out[0].items()}
        host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in dev_out[0].items()}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def e2e_steps(nsteps):
            done = [torch.cuda.Event(), torch.cuda.Event()]     # compute of the step that used buffer b
            landed = [torch.cuda.Event(), torch.cuda.Event()]   # inputs of buffer b copied in
            drained = [torch.cuda.Event(), torch.cuda.Event()]  # results of buffer b copied out
            start = torch.cuda.Event(enable_timing=True)
            stop = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for ev in done + drained:
                ev.record(stream)
            for it in range(nsteps):
                b = it % 2
                s_in.wait_event(done[b])
                with torch.cuda.stream(s_in):
                    for k in names_in:
                        dev_in[b][k].copy_(host_in[k], non_blocking=True)
                    landed[b].record(s_in)
                stream.wait_event(landed[b])
                stream.wait_event(drained[b])
                o = dev_out[b]
                fwd(dev_in[b]["q"], dev_in[b]["k"], dev_in[b]["v"], dev_in[b]["g"], dev_in[b]["beta"], cu_d, cu_host,
                    scale, out=o["out"], ht=ht, saved=saved, save_for_bwd=True)
                bwd(dev_in[b]["q"], dev_in[b]["k"], dev_in[b]["v"], dev_in[b]["g"], dev_in[b]["beta"], cu_d, cu_host,
                    scale, dev_in[b]["dout"], saved, scratch=scratch, grads={k: o[k] for k in grads})
                done[b].record(stream)
                s_out.wait_event(done[b])
                with torch.cuda.stream(s_out):
                    for k in host_out:
                        host_out[k].copy_(o[k], non_blocking=True)
                    drained[b].record(s_out)
            for ev in drained:
                stream.wait_event(ev)
            stop.record(stream)
            barrier()
            return start.elapsed_time(stop) / nsteps

        e2e_steps(2)  # warm-up
        ksteps = max(args.steps // 2, 4)
        e_ms = e2e_steps(ksteps)
        if world > 1:
            tt = torch.tensor([e_ms], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            e_ms = float(tt.item())
        e2e = {"value": world * T / (e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms, "steps": ksteps,
               "pipelined": "inputs of step s+1 copied in and results of step s-1 copied out while step s computes"}
        del host_in, host_out, dev_in, dev_out

    # ---- roofline of the dominant kernel ------------------------------------
    pk = peaks()
    # The dominant kernel: the one that moves the most algorithmic bytes per call.
    # (Launch durations of different document groups overlap one another on
    # their streams, so the largest summed duration would pick the kernel that
    # waits longest for SMs, not the one with the most work.)
    modeled = [name for name in kern if name in KERNEL_MODEL]
    top = max(modeled, key=lambda nm: KERNEL_MODEL[nm][0] * kern[nm][2]) if modeled else None
    roofline = None
    kernels = {}
    # A kernel may run as one launch per document group per call (groups on
    # streams of their own can overlap): bytes per launch = the model's bytes
    # per (token, value head) x the token-heads of the launch.
    for name, (n, ms, units_all) in kern.items():
        avg_ms = ms / n
        entry = {"launches": n, "total_ms": ms, "avg_ms": avg_ms, "share": ms / max(sum(v[1] for v in kern.values()), 1e-9),
                 "ms_per_call": ms / args.steps}
        if name in KERNEL_MODEL:
            b_th, f_th = KERNEL_MODEL[name]
            units = units_all / n
            bytes_ = b_th * units
            flops = f_th * units
            gbs = bytes_ / (avg_ms / 1e3) / 1e9
            tfs = flops / (avg_ms / 1e3) / 1e12
            # TF32 tensor peak = measured BF16 peak x the nominal TF32/BF16 ratio (1.1 / 2.25).
            tf32_peak = pk["bf16_tflops"] * (1.1 / 2.25)
            entry.update(alg_bytes=bytes_, alg_flops=flops, gbs=gbs, tflops=tfs,
                         hbm_frac=gbs / pk["hbm_gbs"], tensor_frac=tfs / tf32_peak)
        kernels[name] = entry
    if top is not None and "hbm_frac" in kernels[top]:
        k = kernels[top]
        tf32_peak = pk["bf16_tflops"] * (1.1 / 2.25)
        if k["hbm_frac"] >= k["tensor_frac"]:
            roofline = {"kernel": top, "bound": "hbm", "achieved": k["gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": k["hbm_frac"], "peak_source": pk["source"]}
        else:
            roofline = {"kernel": top, "bound": "tensor", "achieved": k["tflops"], "peak": tf32_peak,
                        "unit": "TFLOP/s", "frac": k["tensor_frac"],
                        "peak_source": pk["source"] + " bf16 x nominal tf32/bf16 ratio"}
        per_th = ncu_traffic(top)
        roofline["traffic"] = None if per_th is None else per_th * kern[top][2] / kern[top][0]
        roofline["alg_bytes_per_launch"] = k["alg_bytes"]

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1) ------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xh = {k: v.cpu() for k, v in x.items()}
        toks = 4096
        n, dt, threads = oracle_sample(wl, xh, toks)
        cpu = {"value": n / dt / HV, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"first {toks} tokens of each of the {len(wl.lengths)} documents, all {HV} heads, "
                         f"fwd+bwd ({n} token-heads, {dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "tf32", "data": "synthetic",
            "config": {"workload": wl.name, "variant": wl.variant, "T": T, "Hqk": Hqk, "HV": HV, "D": D,
                       "docs": list(wl.lengths), "l2": "inputs larger than L2; 256 MiB flush between steps",
                       "parallelism": f"replicas x{world}"},
            "fwd_ms": statistics.mean(t_fwd), "bwd_ms": statistics.mean(t_bwd), "ckpt_ms": ckpt_ms,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": gpu_launches, "kernels": kernels, "wall_s_timed": wall,
            "kernel_timing": "CUDA events around each launch on its own stream, timed region; launches of "
                             "different document groups run on separate streams and overlap",
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
