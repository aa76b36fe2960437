"""FP64 CPU oracle for the gated delta rule (KDA and GDN) over packed documents.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) use it.  It shares no code with the CUDA
library in ``gated_delta_rule_varlen_gb300``; the only code both sides use is
the seeded input generator in ``synth``, which holds none of the method's
arithmetic.

The arithmetic lives in ``gdr_oracle.cpp`` (a plain FP64 token-by-token
recurrence with a hand-derived reverse pass, threaded over (document, Q/K head)
units).  This module compiles it with the host C++ compiler and marshals numpy
float64 arrays through ctypes.

Sources of the definition: flashinfer PR #8218 "feat(cake_kda): ... Cake KDA
context-parallel (KCP) autograd backend", opening description and "Workload"
paragraph (KDA: per-channel pre-activated log-decay, packed varlen, D=128), and
PR #7723 "perf(cake_gdn): prefetch offset adjoint walk, default LPT segment
plan", opening description (GDN: scalar log-decay, grouped Q/K heads, dq/dk
summed over each Q/K head's value heads).

Pins (tests/test_oracle_pins.py): central finite differences of every
gradient on tiny problems, packed == per-document, the delta-rule write
invariant, one-token closed forms, the g=0 orthonormal-key reduction to causal
linear attention, and KDA <-> GDN equivalences.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle_gdr.so")
_lock = threading.Lock()
_lib = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64),
        ("N", ctypes.c_int32),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
        ("Hqk", ctypes.c_int32),
        ("HV", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("gate_per_channel", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p),
        ("beta", ctypes.c_void_p),
        ("h0", ctypes.c_void_p),
        ("dout", ctypes.c_void_p),
        ("dht", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("ht", ctypes.c_void_p),
        ("dq", ctypes.c_void_p),
        ("dk", ctypes.c_void_p),
        ("dv", ctypes.c_void_p),
        ("dg", ctypes.c_void_p),
        ("dbeta", ctypes.c_void_p),
        ("dh0", ctypes.c_void_p),
        ("threads", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile gdr_oracle.cpp into liboracle_gdr.so next to it (idempotent)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.gdr_oracle_run.argtypes = [ctypes.POINTER(_Problem)]
            lib.gdr_oracle_run.restype = ctypes.c_int
            lib.gdr_oracle_hardware_threads.argtypes = []
            lib.gdr_oracle_hardware_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def hardware_threads() -> int:
    return int(_load().gdr_oracle_hardware_threads())


def _f64(x):
    if x is None:
        return None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# In-kernel q/k L2 normalization (the pages' ``use_qk_l2norm_in_kernel``,
# flashinfer PR #8638 "perf(cake_gdn_kcp): ... graph-replay checkpoint
# recompute hands its tapes to the backward", workload description): each
# (token, Q/K head) vector x of q and of k enters the recurrence as
#     n = x * r,   r = (sum_c x_c^2 + L2NORM_EPS)^(-1/2).
# The pages give the flag but not the formula; this reading (a reciprocal
# square root with a small additive epsilon, so that a zero vector stays
# zero) is recorded with the others.  Its adjoint: with dn the gradient of
# the normalized vector,
#     dx = r * (dn - n * (n . dn)).
L2NORM_EPS = 1e-6


def l2norm(x):
    """(n, r) for x [T, H, D]: the normalized vectors and their scales r [T, H]."""
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt((x * x).sum(-1) + L2NORM_EPS)
    return x * r[..., None], r


def l2norm_backward(n, r, dn):
    """dx from the normalized vectors n, their scales r and the gradient dn."""
    return r[..., None] * (dn - n * (n * dn).sum(-1, keepdims=True))


def run(q, k, v, g, beta, cu_seqlens, scale, h0=None, dout=None, dht=None, threads=0, qk_l2norm=False):
    """Run the oracle.

    Shapes: q, k [T, Hqk, D]; v [T, HV, D]; g [T, HV, D] (KDA, per-channel gate)
    or [T, HV] (GDN, scalar gate); beta [T, HV]; cu_seqlens [N+1] int;
    h0 / dht [N, HV, D, D] or None; dout [T, HV, D] or None (forward only).
    qk_l2norm: normalize q and k first (``l2norm``); dq, dk are then the
    gradients with respect to the raw q, k.

    Returns a dict with ``out`` and ``ht`` and, when ``dout`` is given,
    ``dq dk dv dg dbeta`` and ``dh0`` (the latter only when ``h0`` is given).
    All arrays float64.
    """
    if qk_l2norm:
        qn, rq = l2norm(q)
        kn, rk = l2norm(k)
        res = run(qn, kn, v, g, beta, cu_seqlens, scale, h0=h0, dout=dout, dht=dht, threads=threads)
        if dout is not None:
            res["dq"] = l2norm_backward(qn, rq, res["dq"])
            res["dk"] = l2norm_backward(kn, rk, res["dk"])
        return res
    lib = _load()
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    h0, dout, dht = _f64(h0), _f64(dout), _f64(dht)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T, Hqk, D = q.shape
    HV = v.shape[1]
    N = cu.shape[0] - 1
    if k.shape != q.shape or v.shape != (T, HV, D) or beta.shape != (T, HV):
        raise ValueError("oracle: shape mismatch")
    if g.shape == (T, HV, D):
        per_channel = 1
    elif g.shape == (T, HV):
        per_channel = 0
    else:
        raise ValueError("oracle: gate must be [T,HV,D] or [T,HV]")
    res = {"out": np.zeros((T, HV, D)), "ht": np.zeros((N, HV, D, D))}
    if dout is not None:
        res.update(
            dq=np.zeros((T, Hqk, D)), dk=np.zeros((T, Hqk, D)), dv=np.zeros((T, HV, D)),
            dg=np.zeros(g.shape), dbeta=np.zeros((T, HV)),
        )
        if h0 is not None:
            res["dh0"] = np.zeros((N, HV, D, D))
    p = _Problem()
    p.T, p.N = T, N
    p.cu_seqlens = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    p.Hqk, p.HV, p.D = Hqk, HV, D
    p.gate_per_channel = per_channel
    p.scale = float(scale)
    p.q, p.k, p.v, p.g, p.beta = (_ptr(x) for x in (q, k, v, g, beta))
    p.h0, p.dout, p.dht = _ptr(h0), _ptr(dout), _ptr(dht)
    p.out, p.ht = _ptr(res["out"]), _ptr(res["ht"])
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        setattr(p, name, _ptr(res.get(name)))
    p.threads = int(threads)
    rc = lib.gdr_oracle_run(ctypes.byref(p))
    if rc != 0:
        raise ValueError(f"oracle: invalid problem (rc={rc})")
    return res
