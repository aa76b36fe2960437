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
# The five workloads whose fwd, bwd and ckpt are reported in the line's "configs".
CONFIGS = ("kda_tiny", "kda_pack_h4", "kda_pack_h16", "kda_pack_h64", "gdn_p1", "gdn_1doc")
UNIT = "tokens/s"

# Algorithmic bytes and FLOPs per (token, value head) of each kernel: every
# input read once and every output written once at its stored precision
# (BF16 I/O, FP32 gates and intermediates), and the chunk-64 matrix products
# counted at 2 flops per multiply-add (triangular 64x64 factors at half).
C, D = 64, 128
_TILE = D * 4           # one FP32 row of a [64][128] intermediate
_STATE = D * D * 4 / C  # one FP32 128x128 state per chunk, per token
KERNEL_MODEL = {
    # name: (bytes per token-head, flops per token-head).  w, u, Q Gamma, Kd^T
    # and Aqk are stored in FP16 (2 bytes), the other intermediates in FP32.
    "prep": (3 * 2 * D + 4 * D + 2 + 4 * 2 * D + C * 2 + 2 * C * 4 + 4 * D / C,
             2 * (2 * 0.5 * C * D) + 2 * (2 * 0.5 * C * D) + C * C / 3),
    # state walk with the outputs: reads w, u, Kd^T, Q Gamma, Aqk, gamma; writes
    # Delta, the BF16 state tape and the BF16 output.
    "walk_fwd": (4 * 2 * D + C * 2 + 4 * D / C + _TILE + _STATE / 2 + 2 * D,
                 3 * (2 * D * D) + 2 * 0.5 * C * D),
    "walk_bwd": (C * 2 + 3 * 2 * D + 2 * D + _STATE / 2 + _TILE, 2 * (2 * D * D) + 2 * D * D + 2 * 0.5 * C * D),
    "grad_state": (2 * D + _STATE + 2 * _TILE + 3 * _TILE + 4 * D / C + C * 4, 3 * (2 * D * D)),
    "grad": (3 * 2 * D + 4 * D + 2 + 2 * D + 2 * D + 2 * D + _TILE + 3 * C * 4 + 2 * _TILE + 3 * _TILE + 3 * 2 * D + 4 * D + 2,
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
    ap.add_argument("--no-configs", action="store_true")
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


# Minimal I/O of one call (the algorithmic bytes of the binding roofline):
# every input read once and every output written once, per token (all heads).
def io_bytes(variant: str, Hqk: int, HV: int):
    qk = 2 * Hqk * D * 2
    vrow = HV * D * 2
    gate = HV * D * 4 if variant == "kda" else HV * 4
    beta = HV * 2 if variant == "kda" else HV * 4
    fwd = qk + vrow + gate + beta + vrow                      # q, k, v, g, beta -> out
    bwd = (qk + vrow + gate + beta + vrow) + (qk + vrow + gate + beta)  # + dout -> dq, dk, dv, dg, dbeta
    return fwd, bwd


# Chunked-algorithm flops per (token, value head) (the chunk-64 products of
# the forward and backward as counted in the design notes): forward 140.6
# kflop, backward 282.6 kflop.  GDN shares its Gram products across the
# value heads of a Q/K head; the KDA count is used for it too (an upper bound).
FLOPS_FWD, FLOPS_BWD = 140.6e3, 282.6e3


def binding_roofline(variant, T, Hqk, HV, ms, pk, kind="fwd+bwd"):
    fb, bb = io_bytes(variant, Hqk, HV)
    per_tok = {"fwd": fb, "bwd": bb, "fwd+bwd": fb + bb, "ckpt": 2 * fb + bb}[kind]
    per_th_fl = {"fwd": FLOPS_FWD, "bwd": FLOPS_BWD, "fwd+bwd": FLOPS_FWD + FLOPS_BWD,
                 "ckpt": 2 * FLOPS_FWD + FLOPS_BWD}[kind]
    nbytes = per_tok * T
    flops = per_th_fl * T * HV
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops_sustained"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    return {"bound": bound, "alg_bytes": nbytes, "alg_flops": flops, "t_hbm_ms": 1e3 * t_hbm, "t_tc_ms": 1e3 * t_tc,
            "frac": 1e3 * max(t_hbm, t_tc) / ms}


class Workload:
    """Device inputs, outputs and workspaces of one workload, and its calls."""

    def __init__(self, name, dev, seed=0):
        import torch
        import gated_delta_rule_varlen_gb300 as gdr
        import synth
        self.wl = wl = synth.workload(name)
        self.T, self.Hqk, self.HV = wl.T, wl.Hqk, wl.HV
        self.cu_host = wl.cu_seqlens
        self.x = synth.make_inputs(wl.variant, wl.T, wl.Hqk, wl.HV, D, seed=seed, device=dev)
        self.cu_d = torch.tensor(self.cu_host, dtype=torch.int32, device=dev)
        self.scale = D ** -0.5
        kda = wl.variant == "kda"
        self.fwd = gdr.kda_fwd if kda else gdr.gdn_fwd
        self.bwd = gdr.kda_bwd if kda else gdr.gdn_bwd
        wsb = (gdr.kda_workspace_bytes(wl.T, wl.HV, self.cu_host) if kda
               else gdr.gdn_workspace_bytes(wl.T, wl.Hqk, wl.HV, self.cu_host))
        self.saved = torch.empty(wsb[0], dtype=torch.uint8, device=dev)
        self.scratch = torch.empty(max(wsb), dtype=torch.uint8, device=dev)
        x = self.x
        self.out = torch.empty((wl.T, wl.HV, D), dtype=torch.bfloat16, device=dev)
        self.ht = torch.empty((len(wl.lengths), wl.HV, D, D), dtype=torch.float32, device=dev)
        self.grads = {"dq": torch.empty_like(x["q"]), "dk": torch.empty_like(x["k"]), "dv": torch.empty_like(x["v"]),
                      "dg": torch.empty_like(x["g"]), "dbeta": torch.empty_like(x["beta"])}

    def fwd_call(self, save=True, xx=None, out=None):
        xx = xx or self.x
        return self.fwd(xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], self.cu_d, self.cu_host, self.scale,
                        out=self.out if out is None else out, ht=self.ht, saved=self.saved if save else None,
                        save_for_bwd=save, scratch=None if save else self.scratch)

    def bwd_call(self, xx=None, grads=None):
        xx = xx or self.x
        return self.bwd(xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], self.cu_d, self.cu_host, self.scale,
                        xx["dout"], self.saved, scratch=self.scratch, grads=self.grads if grads is None else grads)


def time_steps(w, stream, flush, nsteps, ckpt=False):
    """Per-step CUDA-event times (ms) of fwd(save) + bwd (fwd and bwd split),
    or of the ckpt sequence fwd(no save) + fwd(save) + bwd; L2 flushed before
    each step (outside the events)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(nsteps)]
    for e0, e1, e2 in evs:
        flush.zero_()
        e0.record(stream)
        if ckpt:
            w.fwd_call(save=False)
        w.fwd_call()
        e1.record(stream)
        w.bwd_call()
        e2.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b, _ in evs], [b.elapsed_time(c) for _, b, c in evs]


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    import gated_delta_rule_varlen_gb300 as gdr

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    gdr.load()
    pk = peaks()

    w = Workload(args.workload, dev)
    wl, T, Hqk, HV, x = w.wl, w.T, w.Hqk, w.HV, w.x
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 1)):
        w.fwd_call()
        w.bwd_call()
    barrier()

    # ---- timed region: K steps of fwd + bwd, no instrumentation ------------
    # The K steps are split into up to 5 consecutive groups; the step time is
    # the median over all K, and the drift is the largest deviation of a
    # group's median from it.
    sampler = ClockSampler(local)
    sampler.start()
    launches0 = gdr.gdr_launch_count()
    barrier()
    wall0 = time.perf_counter()
    t_fwd, t_bwd = time_steps(w, stream, flush, args.steps)
    barrier()
    wall = time.perf_counter() - wall0
    gpu_launches = gdr.gdr_launch_count() - launches0
    clocks = sampler.stop()
    t_step = [f + b for f, b in zip(t_fwd, t_bwd)]
    ms_step = statistics.median(t_step)
    ngroups = min(5, len(t_step))
    per = len(t_step) // ngroups
    group_medians = [statistics.median(t_step[i * per:(i + 1) * per]) for i in range(ngroups)]
    drift = max(abs(m - ms_step) for m in group_medians) / ms_step
    if world > 1:
        tt = torch.tensor([ms_step], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_step = float(tt.item())
    value = world * T / (ms_step / 1e3)

    # ---- ckpt: forward (no save), forward (save), backward -----------------
    ckpt_ms = None
    if not args.no_ckpt:
        barrier()
        cf, cb = time_steps(w, stream, flush, max(args.steps // 4, 3), ckpt=True)
        ckpt_ms = statistics.median([f + b for f, b in zip(cf, cb)])

    # ---- per-kernel times: a separate pass with every launch on the caller's
    # stream (no overlap between document groups) and CUDA events around each.
    barrier()
    prev_serial = gdr.gdr_set_serial(True)
    gdr.gdr_profile_enable(True)
    nprof = 3
    sf, sb = time_steps(w, stream, flush, nprof)
    gdr.gdr_profile_enable(False)
    gdr.gdr_set_serial(prev_serial)
    kern = gdr.gdr_profile_report()
    serial_ms = statistics.median([f + b for f, b in zip(sf, sb)])
    kernels = {}
    tf32_peak = pk["bf16_tflops"] * (1.1 / 2.25)  # measured BF16 x the nominal TF32/BF16 ratio
    total_kms = max(sum(v[1] for v in kern.values()), 1e-9)
    for name, (n, ms, units_all) in kern.items():
        avg_ms = ms / n
        entry = {"launches_per_step": n / nprof, "ms_per_step": ms / nprof, "avg_launch_ms": avg_ms,
                 "share": ms / total_kms}
        if name in KERNEL_MODEL:
            b_th, f_th = KERNEL_MODEL[name]
            units = units_all / n
            gbs = b_th * units / (avg_ms / 1e3) / 1e9
            tfs = f_th * units / (avg_ms / 1e3) / 1e12
            per_th = ncu_traffic(name)
            entry.update(design_bytes_per_token_head=b_th, gbs=gbs, tflops=tfs, hbm_frac=gbs / pk["hbm_gbs"],
                         tf32_frac=tfs / tf32_peak,
                         ncu_bytes_per_token_head=per_th,
                         traffic_over_design=None if per_th is None else per_th / b_th)
        kernels[name] = entry
    # The dominant kernel: the largest share of the serialized kernel time.
    top = max(kern, key=lambda nm: kern[nm][1]) if kern else None
    top_roofline = None
    if top is not None and "gbs" in kernels[top]:
        k = kernels[top]
        n, ms, units_all = kern[top]
        units = units_all / n
        per_th = k["ncu_bytes_per_token_head"]
        if k["hbm_frac"] >= k["tf32_frac"]:
            top_roofline = {"kernel": top, "bound": "hbm", "achieved": k["gbs"], "peak": pk["hbm_gbs"],
                            "unit": "GB/s", "frac": k["hbm_frac"]}
        else:
            top_roofline = {"kernel": top, "bound": "tensor", "achieved": k["tflops"], "peak": tf32_peak,
                            "unit": "TFLOP/s", "frac": k["tf32_frac"]}
        top_roofline.update(share=k["share"], alg_bytes_per_launch=KERNEL_MODEL[top][0] * units,
                            traffic=None if per_th is None else per_th * units,
                            bytes_model="the kernel's own inputs read once and outputs written once at their "
                                        "stored precision (bench.KERNEL_MODEL)")

    # ---- the whole step against the binding roofline: max(bytes / HBM, flops / BF16) ----
    rf = binding_roofline(wl.variant, T, Hqk, HV, ms_step, pk)
    traffic = None
    if all(kernels.get(nm, {}).get("ncu_bytes_per_token_head") is not None for nm in kernels if nm in KERNEL_MODEL):
        per_th = sum(kernels[nm]["ncu_bytes_per_token_head"] for nm in kernels if nm in KERNEL_MODEL)
        traffic = per_th * T * HV if per_th else None
    roofline = {"bound": rf["bound"], "achieved": rf["alg_bytes"] / (ms_step / 1e3) / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": rf["frac"], "traffic": traffic, "alg_bytes_per_step": rf["alg_bytes"],
                "alg_flops_per_step": rf["alg_flops"], "t_hbm_ms": rf["t_hbm_ms"], "t_tc_ms": rf["t_tc_ms"],
                "peak_source": pk["source"], "scope": "whole fwd+bwd step: minimal I/O at HBM bandwidth vs "
                "chunked-algorithm flops at the sustained BF16 peak, over the median step time"}
    if rf["bound"] == "tensor":
        roofline.update(achieved=rf["alg_flops"] / (ms_step / 1e3) / 1e12, peak=pk["bf16_tflops_sustained"],
                        unit="TFLOP/s")

    # ---- end to end through the C ABI with host buffers --------------------
    # Every step copies its inputs from pinned host memory and its results
    # (out and every gradient) back.  Steps are pipelined the way a training
    # loop with host-resident data runs them: device inputs and outputs are
    # double-buffered, step s+1's inputs are copied in and step s-1's results
    # copied out while step s computes, each direction on two copy streams
    # (each tensor in two contiguous halves: two streams per direction move
    # ~7% more than one over the host link when both directions run).  The
    # timed region runs from before the first input copy to after the last
    # result copy.
    e2e = None
    if not args.no_e2e:
        names_in = ("q", "k", "v", "g", "beta", "dout")
        host_in = {k: x[k].cpu().pin_memory() for k in names_in}
        dev_in = [{k: x[k] for k in names_in}, {k: torch.empty_like(x[k]) for k in names_in}]
        dev_out = [{"out": w.out, **w.grads}, None]
        dev_out[1] = {k: torch.empty_like(v) for k, v in dev_out[0].items()}
        host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in dev_out[0].items()}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        NCS = 2  # copy streams per direction
        s_in = [torch.cuda.Stream() for _ in range(NCS)]
        s_out = [torch.cuda.Stream() for _ in range(NCS)]

        def half(t, i):  # contiguous part i of NCS of a tensor, flattened
            f = t.view(-1)
            n = (f.numel() + NCS - 1) // NCS
            return f[i * n:(i + 1) * n]

        def e2e_steps(nsteps):
            done = [torch.cuda.Event(), torch.cuda.Event()]  # compute of the step that used buffer b
            landed = [[torch.cuda.Event() for _ in range(NCS)] for _ in range(2)]   # inputs of buffer b in
            drained = [[torch.cuda.Event() for _ in range(NCS)] for _ in range(2)]  # results of buffer b out
            start = torch.cuda.Event(enable_timing=True)
            stop = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for ev in done + drained[0] + drained[1]:
                ev.record(stream)
            for it in range(nsteps):
                b = it % 2
                for i in range(NCS):
                    s_in[i].wait_event(done[b])
                    with torch.cuda.stream(s_in[i]):
                        for k in names_in:
                            half(dev_in[b][k], i).copy_(half(host_in[k], i), non_blocking=True)
                        landed[b][i].record(s_in[i])
                for i in range(NCS):
                    stream.wait_event(landed[b][i])
                    stream.wait_event(drained[b][i])
                o = dev_out[b]
                w.fwd_call(xx=dev_in[b], out=o["out"])
                w.bwd_call(xx=dev_in[b], grads={k: o[k] for k in w.grads})
                done[b].record(stream)
                for i in range(NCS):
                    s_out[i].wait_event(done[b])
                    with torch.cuda.stream(s_out[i]):
                        for k in host_out:
                            half(host_out[k], i).copy_(half(o[k], i), non_blocking=True)
                        drained[b][i].record(s_out[i])
            for ev in drained[0] + drained[1]:
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

    headline = {"fwd_ms": statistics.median(t_fwd), "bwd_ms": statistics.median(t_bwd), "ckpt_ms": ckpt_ms}

    # ---- every configuration: fwd, bwd, ckpt, tokens/s, binding fraction ----
    configs = None
    if not args.no_configs:
        configs = {}
        for name in CONFIGS:
            if name == args.workload:
                c = dict(headline, steps=args.steps)
                fms, bms, cms = headline["fwd_ms"], headline["bwd_ms"], ckpt_ms
                cw = w
            else:
                cw = Workload(name, dev)
                for _ in range(2):
                    cw.fwd_call()
                    cw.bwd_call()
                nst = max(3, args.steps // 4)
                f_, b_ = time_steps(cw, stream, flush, nst)
                cf, cb = time_steps(cw, stream, flush, max(2, nst // 2), ckpt=True)
                fms, bms = statistics.median(f_), statistics.median(b_)
                cms = statistics.median([p + q for p, q in zip(cf, cb)])
                c = {"fwd_ms": fms, "bwd_ms": bms, "ckpt_ms": cms, "steps": nst}
            c.update(tokens_per_s=cw.T / ((fms + bms) / 1e3), T=cw.T, Hqk=cw.Hqk, HV=cw.HV,
                     docs=len(cw.wl.lengths),
                     frac_fwd_bwd=binding_roofline(cw.wl.variant, cw.T, cw.Hqk, cw.HV, fms + bms, pk)["frac"],
                     frac_fwd=binding_roofline(cw.wl.variant, cw.T, cw.Hqk, cw.HV, fms, pk, "fwd")["frac"],
                     frac_bwd=binding_roofline(cw.wl.variant, cw.T, cw.Hqk, cw.HV, bms, pk, "bwd")["frac"],
                     frac_ckpt=(None if cms is None else
                                binding_roofline(cw.wl.variant, cw.T, cw.Hqk, cw.HV, cms, pk, "ckpt")["frac"]))
            configs[name] = c
            if cw is not w:
                del cw
                torch.cuda.empty_cache()

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1) ------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xh = {k: v.cpu() for k, v in x.items()}
        # A bounded sample of about 10-30 s of CPU work: a 4096-token probe,
        # then, if it ran short, a longer prefix of every document sized to ~12 s.
        toks = 4096
        n, dt, threads = oracle_sample(wl, xh, toks)
        if dt < 8.0 and toks < max(wl.lengths):
            toks = min(max(wl.lengths), int(toks * 12.0 / max(dt, 1e-3)))
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
            **headline,
            "timing": {"statistic": "median of per-step CUDA-event times", "mean_ms": statistics.mean(t_step),
                       "groups": ngroups, "group_medians_ms": group_medians, "drift": drift},
            "roofline": roofline, "top_kernel_roofline": top_roofline, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks, "gpu_launches": gpu_launches, "configs": configs, "kernels": kernels,
            "kernel_timing": f"separate pass of {nprof} steps with every launch on the caller's stream "
                             f"(document groups serialized; {serial_ms:.2f} ms per step), CUDA events around "
                             "each launch; shares are of the summed kernel time",
            "wall_s_timed": wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
