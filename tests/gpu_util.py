"""Helpers for the GPU parity tests: run the CUDA path through the binding and
the FP64 oracle on the same seeded inputs, and compare.

Tolerances (relative L2 over the whole compared tensor): out and ht 3e-3,
every gradient (dq, dk, dv, dg, dbeta, dh0) 1e-2.  Each comparison also
reports the max-abs error max|x - ref| and the same divided by max|ref|, and
the fraction of elements outside the elementwise bound |x - ref| <= 1e-2 +
1e-2 |ref| (the acceptance clause of PR #7723's accuracy gates), for
information: only the relative L2 is asserted.
"""
import numpy as np
import torch

import oracle

TOL = {"out": 3e-3, "ht": 3e-3, "dq": 1e-2, "dk": 1e-2, "dv": 1e-2, "dg": 1e-2, "dbeta": 1e-2, "dh0": 1e-2}
SCALE = 128 ** -0.5


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    if nb == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def f64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def run_gpu(variant, x, cu, scale=SCALE, h0=None, dht=None, backward=True, want_dh0=False, dev="cuda", l2=False):
    import gated_delta_rule_varlen_gb300 as gdr

    xd = {k: v.to(dev) for k, v in x.items()}
    cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
    h0d = None if h0 is None else h0.to(dev)
    dhtd = None if dht is None else dht.to(dev)
    fwd = gdr.kda_fwd if variant == "kda" else gdr.gdn_fwd
    bwd = gdr.kda_bwd if variant == "kda" else gdr.gdn_bwd
    # Outputs and workspaces start as NaN (workspace bytes 0xFF: a NaN in FP32
    # and BF16), so a read of memory nothing wrote shows up in the comparison.
    T, Hqk, D = xd["q"].shape
    HV, N = xd["v"].shape[1], len(cu) - 1
    if variant == "kda":
        sb, cb = gdr.kda_workspace_bytes(T, HV, cu, l2)
    else:
        sb, cb = gdr.gdn_workspace_bytes(T, Hqk, HV, cu, l2)
    poison = lambda n: torch.full((max(int(n), 256),), 0xFF, dtype=torch.uint8, device=dev)
    nan = float("nan")
    out = torch.full((T, HV, D), nan, dtype=torch.bfloat16, device=dev)
    ht = torch.full((N, HV, D, D), nan, dtype=torch.float32, device=dev)
    out, ht, saved = fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, scale, h0=h0d, out=out, ht=ht,
                         saved=poison(sb) if backward else None, scratch=None if backward else poison(sb),
                         save_for_bwd=backward, qk_l2norm=l2)
    res = {"out": out, "ht": ht}
    if backward:
        grads = {n: torch.full_like(xd[src], nan) for n, src in
                 (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"))}
        if want_dh0:
            grads["dh0"] = torch.full((N, HV, D, D), nan, dtype=torch.float32, device=dev)
        res.update(bwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, scale, xd["dout"], saved, h0=h0d,
                       dht=dhtd, want_dh0=want_dh0, scratch=poison(cb), grads=grads, qk_l2norm=l2))
    torch.cuda.synchronize()
    gdr.gdr_check_device()  # no kernel gave up a bounded wait
    return res


def run_oracle(x, cu, scale=SCALE, h0=None, dht=None, backward=True, l2=False):
    f = {k: f64(v) for k, v in x.items()}
    return oracle.run(f["q"], f["k"], f["v"], f["g"], f["beta"], cu, scale, h0=f64(h0),
                      dout=f["dout"] if backward else None, dht=f64(dht), qk_l2norm=l2)


class Err(float):
    """Relative L2 error (the float value, which the tolerances apply to) with
    the max-abs error, max|ref| and the elementwise-clause miss fraction."""

    def __new__(cls, r, max_abs, max_ref, miss):
        e = super().__new__(cls, r)
        e.max_abs, e.max_ref, e.miss = max_abs, max_ref, miss
        return e

    def __repr__(self):
        return (f"rel={float(self):.3e} maxabs={self.max_abs:.3e} "
                f"(/max|ref| {self.max_abs / max(self.max_ref, 1e-300):.3e}) miss1e-2={self.miss:.1e}")


def err_stats(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    d = np.abs(a - b)
    max_abs = float(d.max()) if d.size else 0.0
    max_ref = float(np.abs(b).max()) if b.size else 0.0
    miss = float(np.mean(d > 1e-2 + 1e-2 * np.abs(b))) if d.size else 0.0
    return Err(rel(a, b), max_abs, max_ref, miss)


def compare(gpu, ref, names=None):
    names = names or [n for n in TOL if n in gpu and n in ref and gpu[n] is not None]
    errs = {}
    for n in names:
        errs[n] = err_stats(f64(gpu[n]) if torch.is_tensor(gpu[n]) else gpu[n], ref[n])
    return errs


def assert_within(errs, tol=TOL):
    bad = {k: float(v) for k, v in errs.items() if not (v <= tol[k])}
    msg = " | ".join(f"{k}: {v!r}" if isinstance(v, Err) else f"{k}: rel={v:.3e}" for k, v in errs.items())
    assert not bad, f"parity failed: {bad} (all: {msg})"
    return msg
