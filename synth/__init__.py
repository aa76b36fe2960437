"""Seeded synthetic inputs for the gated delta rule workloads.

This module is the one piece of code that both the CUDA path's tests/bench and
the FP64 oracle consume.  It holds none of the method's arithmetic: it only
draws random tensors in the shapes, dtypes and distributions of the workloads
and builds the packed-document offsets.

Workloads (what the pages time; "Workload" paragraph of flashinfer PR #8218
"feat(cake_kda): ... Cake KDA context-parallel (KCP) autograd backend", and the
pack table of PR #7723 "perf(cake_gdn): prefetch offset adjoint walk, default
LPT segment plan"):

* KDA: one packed batch of 4 documents, 42024 / 57573 / 73122 / 88673 tokens
  (T = 261392), H in {4, 16, 64}, D = 128.  q, k, v BF16 [T, H, 128] with q and
  k L2-normalized per (token, head) vector; g FP32 [T, H, 128] uniform in
  (-5, 0) (pre-activated log-decay); beta BF16 [T, H] uniform in (0, 1).
* KDA tiny: one document of 512 tokens, H = 1.
* GDN: (H_qk, HV) = (16, 48), D = 128; q, k BF16 [T, 16, 128] L2-normalized;
  v BF16 [T, 48, 128]; g and beta FP32 [T, 48]; packs of 241817 tokens in 6
  seeded-random documents (the pages do not print P1's document lengths) and
  32768 tokens in one document.

Draw order (fixed so that any consumer reproduces the same tensors from the
seed): q, k, v ~ N(0, 1) in FP32; q and k divided by their L2 norm over the
head dimension in FP32, then rounded to BF16; g ~ U(-5, 0) FP32; beta ~ U(0, 1)
(BF16 for KDA, FP32 for GDN); dout ~ N(0, 1) rounded to BF16.  The generator is
``torch.Generator(device)`` seeded with ``seed``.  The same seed gives the same
numbers on the same device type; CPU and CUDA streams differ, so a test that
compares the two paths draws once and hands the same tensors to both.
"""
from __future__ import annotations

import dataclasses

import torch

KDA_PACK_DOCS = (42024, 57573, 73122, 88673)  # T = 261392
GDN_P1_TOKENS = 241817
GDN_P1_DOCS = 6
GDN_1DOC_TOKENS = 32768


def cu_from_lengths(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return cu


def random_pack_lengths(total: int, ndocs: int, seed: int = 0):
    """Document lengths of a pack of `total` tokens cut at ndocs-1 distinct
    seeded-random points: sorted(randperm(total - 1)[:ndocs - 1] + 1)."""
    if ndocs == 1:
        return [total]
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    cuts = (torch.randperm(total - 1, generator=g)[: ndocs - 1] + 1).sort().values.tolist()
    edges = [0] + cuts + [total]
    return [edges[i + 1] - edges[i] for i in range(ndocs)]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    variant: str  # "kda" or "gdn"
    lengths: tuple
    Hqk: int
    HV: int
    D: int = 128

    @property
    def T(self) -> int:
        return int(sum(self.lengths))

    @property
    def cu_seqlens(self):
        return cu_from_lengths(self.lengths)


def workload(name: str) -> Workload:
    """The named workloads: kda_tiny, kda_pack_h4, kda_pack_h16, kda_pack_h64,
    gdn_p1 (241817 tokens / 6 docs), gdn_1doc (32768 tokens / 1 doc), and the
    profiling-size cases kda_prof (4 x 16384 tokens, H = 4), kda_prof16
    (4 x 4096 tokens, H = 16) and gdn_prof (2 x 4096 tokens, (16, 48))."""
    if name == "kda_tiny":
        return Workload(name, "kda", (512,), 1, 1)
    if name == "kda_prof":  # profiling-size pack: 4 x 16384 tokens, H = 4 (inputs > L2, a few GB in all)
        return Workload(name, "kda", (16384,) * 4, 4, 4)
    if name == "kda_prof16":  # profiling-size pack with H = 16 chains per document: 4 x 4096 tokens, H = 16
        return Workload(name, "kda", (4096,) * 4, 16, 16)
    if name.startswith("kda_pack_h"):
        h = int(name[len("kda_pack_h"):])
        return Workload(name, "kda", KDA_PACK_DOCS, h, h)
    if name == "gdn_p1":
        return Workload(name, "gdn", tuple(random_pack_lengths(GDN_P1_TOKENS, GDN_P1_DOCS, 0)), 16, 48)
    if name == "gdn_1doc":
        return Workload(name, "gdn", (GDN_1DOC_TOKENS,), 16, 48)
    if name == "gdn_prof":  # profiling-size grouped pack: 2 x 4096 tokens, (Hqk, HV) = (16, 48)
        return Workload(name, "gdn", (4096,) * 2, 16, 48)
    raise KeyError(name)


def _l2norm_bf16(x: torch.Tensor) -> torch.Tensor:
    n = x.pow(2).sum(-1, keepdim=True).sqrt().clamp_min(1e-12)
    return (x / n).to(torch.bfloat16)


def make_inputs(variant: str, T: int, Hqk: int, HV: int, D: int = 128, seed: int = 0,
                device="cpu", gate_low: float = -5.0, gate_high: float = 0.0,
                with_dout: bool = True, normalize_qk: bool = True):
    """Draw one problem's inputs.  Returns a dict of tensors on `device`:
    q, k [T,Hqk,D] bf16; v [T,HV,D] bf16; g [T,HV,D] (kda) or [T,HV] (gdn) fp32;
    beta [T,HV] (bf16 kda, fp32 gdn); dout [T,HV,D] bf16 (when with_dout).
    normalize_qk=False leaves q and k as drawn, N(0,1) rows times a per-row
    factor U(0.25, 4) (raw inputs for the in-kernel L2 normalization)."""
    if variant not in ("kda", "gdn"):
        raise ValueError(variant)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    f32 = dict(dtype=torch.float32, device=device, generator=gen)
    out = {}
    if normalize_qk:
        out["q"] = _l2norm_bf16(torch.randn((T, Hqk, D), **f32))
        out["k"] = _l2norm_bf16(torch.randn((T, Hqk, D), **f32))
    else:
        for name in ("q", "k"):
            x = torch.randn((T, Hqk, D), **f32)
            out[name] = (x * (torch.rand((T, Hqk, 1), **f32) * 3.75 + 0.25)).to(torch.bfloat16)
    out["v"] = torch.randn((T, HV, D), **f32).to(torch.bfloat16)
    gshape = (T, HV, D) if variant == "kda" else (T, HV)
    out["g"] = torch.rand(gshape, **f32) * (gate_high - gate_low) + gate_low
    b = torch.rand((T, HV), **f32)
    out["beta"] = b.to(torch.bfloat16) if variant == "kda" else b
    if with_dout:
        out["dout"] = torch.randn((T, HV, D), **f32).to(torch.bfloat16)
    return out


def make_states(N: int, HV: int, D: int = 128, seed: int = 1, device="cpu", scale: float = 1.0):
    """A random FP32 state [N, HV, D, D] (for h0 / dht), N(0, scale^2)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randn((N, HV, D, D), dtype=torch.float32, device=device, generator=gen) * scale
