"""GB300 (sm_103a) chunked gated delta-rule training: KDA and GDN over packed
variable-length documents, head dimension 128.

This module is a thin ctypes binding over ``lib/libgdr.so`` (the C ABI declared
in ``include/gdr.h``).  It only marshals arguments: torch tensors provide
device memory and the current CUDA stream, and every step of the computation
runs in the library's CUDA kernels.  There is no CPU fallback: if the library
is missing, every call raises.

Entry points carry the C names (``kda_workspace_bytes``, ``kda_fwd``,
``kda_bwd``, ``gdn_workspace_bytes``, ``gdn_fwd``, ``gdn_bwd``,
``gdr_status_string``).  Outputs and workspaces are allocated with torch when
the caller does not pass them.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libgdr.so")

# Status codes (include/gdr.h).
GDR_OK = 0
GDR_INVALID_ARG = 1
GDR_BAD_CU_SEQLENS = 2
GDR_WORKSPACE_TOO_SMALL = 3
GDR_UNSUPPORTED = 4
GDR_STALE_WORKSPACE = 5
GDR_CUDA_ERROR = 6
GDR_DEVICE_TIMEOUT = 7

EXPORTED = (
    "gdr_status_string",
    "kda_workspace_bytes",
    "kda_fwd",
    "kda_bwd",
    "kda_fwd_noalloc",
    "gdn_workspace_bytes",
    "gdn_fwd",
    "gdn_bwd",
    "gdr_profile_enable",
    "gdr_profile_report",
    "gdr_check_device",
    "gdr_inject_device_error",
    "gdr_selftest_wait",
    "gdr_doc_groups",
    "gdr_launch_count",
    "gdr_set_serial",
    "gdr_set_segment_chunks",
    "gdr_set_slice_chunks",
    "gdr_walk_slices",
    "gdr_segment_plan",
)

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
SZ = ctypes.c_size_t
F32 = ctypes.c_float
PI32 = ctypes.POINTER(ctypes.c_int32)
PSZ = ctypes.POINTER(ctypes.c_size_t)

_SIGS = {
    "gdr_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "gdr_profile_enable": ([ctypes.c_int], ctypes.c_int),
    "gdr_check_device": ([], ctypes.c_int),
    "gdr_inject_device_error": ([ctypes.c_int], ctypes.c_int),
    "gdr_selftest_wait": ([ctypes.c_uint64, P], ctypes.c_int),
    "gdr_doc_groups": ([I32, PI32, PI32, ctypes.POINTER(ctypes.c_int64), PI32], ctypes.c_int),
    "gdr_profile_report": ([ctypes.c_char_p, SZ], ctypes.c_int),
    "gdr_launch_count": ([], ctypes.c_uint64),
    "gdr_set_serial": ([ctypes.c_int], ctypes.c_int),
    "gdr_set_segment_chunks": ([ctypes.c_int], ctypes.c_int),
    "gdr_set_slice_chunks": ([ctypes.c_int], ctypes.c_int),
    "gdr_walk_slices": ([I32, I32, PI32, I32, PI32], ctypes.c_int),
    "gdr_segment_plan": ([I32, PI32, I32, PI32, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "kda_workspace_bytes": ([I64, I32, I32, PI32, ctypes.c_int, PSZ, PSZ], ctypes.c_int),
    "gdn_workspace_bytes": ([I64, I32, I32, I32, PI32, ctypes.c_int, PSZ, PSZ], ctypes.c_int),
    "kda_fwd": ([P, P, P, P, P, P, PI32, I32, I64, I32, F32, ctypes.c_int, P, P, P, P, SZ, ctypes.c_int, P, SZ, P],
                ctypes.c_int),
    "kda_bwd": ([P, P, P, P, P, P, PI32, I32, I64, I32, F32, ctypes.c_int, P, P, P, P, SZ, P, P, P, P, P, P, P, SZ,
                 P], ctypes.c_int),
    "kda_fwd_noalloc": ([P, P, P, P, P, P, PI32, I32, I64, I32, F32, P, P, P, P], ctypes.c_int),
    "gdn_fwd": ([P, P, P, P, P, P, PI32, I32, I64, I32, I32, F32, ctypes.c_int, P, P, P, P, SZ, ctypes.c_int, P,
                 SZ, P], ctypes.c_int),
    "gdn_bwd": ([P, P, P, P, P, P, PI32, I32, I64, I32, I32, F32, ctypes.c_int, P, P, P, P, SZ, P, P, P, P, P, P,
                 P, SZ, P], ctypes.c_int),
}


class GdrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load(path: str = LIB_PATH):
    """Load libgdr.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libgdr.so not found at {path}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            for name, (args, res) in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().gdr_status_string(int(status)).decode()


gdr_status_string = status_string


def _check(status: int, where: str):
    if status != GDR_OK:
        if status in (GDR_INVALID_ARG, GDR_BAD_CU_SEQLENS, GDR_WORKSPACE_TOO_SMALL):
            raise ValueError(f"{where}: {status_string(status)}")
        raise GdrError(status, where)


def _cu_host(cu_seqlens_host):
    import numpy as np
    if hasattr(cu_seqlens_host, "detach"):
        cu_seqlens_host = cu_seqlens_host.detach().cpu().numpy()
    arr = np.ascontiguousarray(np.asarray(cu_seqlens_host, dtype=np.int32))
    return arr, arr.ctypes.data_as(PI32)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def kda_workspace_bytes(T: int, H: int, cu_seqlens_host, qk_l2norm: bool = False):
    """(saved_bytes, scratch_bytes) for a KDA problem; host only."""
    arr, p = _cu_host(cu_seqlens_host)
    sb, cb = SZ(0), SZ(0)
    _check(load().kda_workspace_bytes(T, H, arr.shape[0] - 1, p, int(bool(qk_l2norm)), ctypes.byref(sb),
                                      ctypes.byref(cb)), "kda_workspace_bytes")
    return sb.value, cb.value


def gdn_workspace_bytes(T: int, Hqk: int, HV: int, cu_seqlens_host, qk_l2norm: bool = False):
    arr, p = _cu_host(cu_seqlens_host)
    sb, cb = SZ(0), SZ(0)
    _check(load().gdn_workspace_bytes(T, Hqk, HV, arr.shape[0] - 1, p, int(bool(qk_l2norm)), ctypes.byref(sb),
                                      ctypes.byref(cb)), "gdn_workspace_bytes")
    return sb.value, cb.value


def _empty_bytes(n, device):
    import torch
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device=device)


def _check_shapes(variant, q, k, v, g, beta, dout=None):
    """Shapes the C ABI assumes (it receives pointers only): q, k [T, Hqk, 128]; v (and dout)
    [T, HV, 128]; g [T, HV, 128] (KDA) or [T, HV] (GDN); beta [T, HV]; Hqk == HV for KDA."""
    T, Hqk, D = q.shape
    HV = v.shape[1]
    want = {"k": (k, (T, Hqk, D)), "v": (v, (T, HV, D)), "beta": (beta, (T, HV)),
            "g": (g, (T, HV, D) if variant == "kda" else (T, HV))}
    if dout is not None:
        want["dout"] = (dout, (T, HV, D))
    for name, (t, shape) in want.items():
        if tuple(t.shape) != shape:
            raise ValueError(f"{variant}: {name} has shape {tuple(t.shape)}, expected {shape}")
    if D != 128:
        raise ValueError(f"{variant}: head dim {D}, only 128 is supported")
    if variant == "kda" and Hqk != HV:
        raise ValueError(f"kda: q/k have {Hqk} heads and v has {HV}; KDA needs the same count")


def _fwd(variant, q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, h0, out, ht, want_ht, saved,
         save_for_bwd, scratch, stream, qk_l2norm=False):
    import torch
    _check_shapes(variant, q, k, v, g, beta)
    T, Hqk, D = q.shape
    HV = v.shape[1]
    arr, cup = _cu_host(cu_seqlens_host)
    N = arr.shape[0] - 1
    if variant == "kda":
        sb, cb = kda_workspace_bytes(T, HV, arr, qk_l2norm)
    else:
        sb, cb = gdn_workspace_bytes(T, Hqk, HV, arr, qk_l2norm)
    dev = q.device
    if out is None:
        out = torch.empty((T, HV, D), dtype=torch.bfloat16, device=dev)
    if ht is None and want_ht:
        ht = torch.empty((N, HV, D, D), dtype=torch.float32, device=dev)
    if save_for_bwd and saved is None:
        saved = _empty_bytes(sb, dev)
    if saved is None and scratch is None:
        scratch = _empty_bytes(sb, dev)
    lib = load()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), cup, N, T]
    args += [HV] if variant == "kda" else [Hqk, HV]
    args += [float(scale), int(bool(qk_l2norm)), _ptr(h0), _ptr(out), _ptr(ht), _ptr(saved),
             0 if saved is None else saved.numel(), int(bool(save_for_bwd)), _ptr(scratch),
             0 if scratch is None else scratch.numel(), _stream(stream)]
    fn = lib.kda_fwd if variant == "kda" else lib.gdn_fwd
    _check(fn(*args), f"{variant}_fwd")
    return out, ht, saved


def _bwd(variant, q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, dout, saved, h0, dht, want_dh0, scratch,
         grads, stream, qk_l2norm=False):
    import torch
    _check_shapes(variant, q, k, v, g, beta, dout)
    T, Hqk, D = q.shape
    HV = v.shape[1]
    arr, cup = _cu_host(cu_seqlens_host)
    N = arr.shape[0] - 1
    if variant == "kda":
        sb, cb = kda_workspace_bytes(T, HV, arr, qk_l2norm)
    else:
        sb, cb = gdn_workspace_bytes(T, Hqk, HV, arr, qk_l2norm)
    dev = q.device
    grads = dict(grads or {})
    for name, like in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta)):
        if name not in grads:  # allocate only what the caller did not pass
            grads[name] = torch.empty_like(like)
    if want_dh0 and "dh0" not in grads:
        grads["dh0"] = torch.empty((N, HV, D, D), dtype=torch.float32, device=dev)
    if scratch is None:
        scratch = _empty_bytes(cb, dev)
    lib = load()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), cup, N, T]
    args += [HV] if variant == "kda" else [Hqk, HV]
    args += [float(scale), int(bool(qk_l2norm)), _ptr(h0), _ptr(dout), _ptr(dht), _ptr(saved), saved.numel(),
             _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]), _ptr(grads["dg"]), _ptr(grads["dbeta"]),
             _ptr(grads.get("dh0")), _ptr(scratch), scratch.numel(), _stream(stream)]
    fn = lib.kda_bwd if variant == "kda" else lib.gdn_bwd
    _check(fn(*args), f"{variant}_bwd")
    return grads


def kda_fwd(q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, h0=None, out=None, ht=None, want_ht=True,
            saved=None, save_for_bwd=True, scratch=None, stream=None, qk_l2norm=False):
    """KDA forward.  q, k, v bf16 [T,H,128]; g fp32 [T,H,128]; beta bf16 [T,H];
    cu_seqlens int32 device [N+1] and its host copy.  qk_l2norm: normalize q, k
    per (token, head) vector in the kernels (the backward must be called with
    the same flag).  Returns (out, ht, saved)."""
    return _fwd("kda", q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, h0, out, ht, want_ht, saved,
                save_for_bwd, scratch, stream, qk_l2norm)


def kda_bwd(q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, dout, saved, h0=None, dht=None, want_dh0=False,
            scratch=None, grads=None, stream=None, qk_l2norm=False):
    """KDA backward from `saved` (filled by kda_fwd(save_for_bwd=True)).
    Returns a dict with dq, dk, dv, dg, dbeta (and dh0 when want_dh0)."""
    return _bwd("kda", q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, dout, saved, h0, dht, want_dh0,
                scratch, grads, stream, qk_l2norm)


def gdn_fwd(q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, h0=None, out=None, ht=None, want_ht=True,
            saved=None, save_for_bwd=True, scratch=None, stream=None, qk_l2norm=False):
    """GDN forward.  q, k bf16 [T,Hqk,128]; v bf16 [T,HV,128]; g, beta fp32
    [T,HV].  Returns (out, ht, saved)."""
    return _fwd("gdn", q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, h0, out, ht, want_ht, saved,
                save_for_bwd, scratch, stream, qk_l2norm)


def gdn_bwd(q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, dout, saved, h0=None, dht=None, want_dh0=False,
            scratch=None, grads=None, stream=None, qk_l2norm=False):
    return _bwd("gdn", q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, dout, saved, h0, dht, want_dh0,
                scratch, grads, stream, qk_l2norm)


def gdr_launch_count() -> int:
    """Kernel launches the library's compute calls have enqueued since it was loaded."""
    return int(load().gdr_launch_count())


def gdr_set_serial(on: bool) -> bool:
    """Run every call's launches on the caller's stream (document groups in
    turn) while on; returns the previous setting."""
    return bool(load().gdr_set_serial(int(bool(on))))


def gdr_set_segment_chunks(chunks: int) -> int:
    """Force walk segments of about `chunks` chunks (0: the library's choice);
    returns the previous setting."""
    return int(load().gdr_set_segment_chunks(int(chunks)))


def gdr_set_slice_chunks(chunks: int) -> int:
    """Slice length (chunks) of pipelined walks, 0 for the default; returns the previous setting."""
    return int(load().gdr_set_slice_chunks(int(chunks)))


def gdr_profile_enable(on: bool = True):
    """Start (True) or stop (False) per-kernel CUDA-event timing; starting clears old records."""
    load().gdr_profile_enable(int(bool(on)))


def gdr_profile_report():
    """{kernel name: (launches, total_ms, token_heads)} of the launches recorded while
    profiling was on (sums over the launches)."""
    buf = ctypes.create_string_buffer(1 << 16)
    _check(load().gdr_profile_report(buf, len(buf)), "gdr_profile_report")
    out = {}
    for line in buf.value.decode().splitlines():
        name, n, ms, units = line.split()
        out[name] = (int(n), float(ms), float(units))
    return out


def gdr_doc_groups(cu_seqlens_host):
    """[(rank_begin, rank_end, chunk_begin, chunk_end)] of the backward's document
    groups for these cu_seqlens (host-side plan; no device work)."""
    arr, cup = _cu_host(cu_seqlens_host)
    ranks = (ctypes.c_int32 * 5)()
    chunks = (ctypes.c_int64 * 5)()
    n = ctypes.c_int32(0)
    _check(load().gdr_doc_groups(arr.shape[0] - 1, cup, ranks, chunks, ctypes.byref(n)), "gdr_doc_groups")
    return [(ranks[i], ranks[i + 1], chunks[i], chunks[i + 1]) for i in range(n.value)]


def gdr_segment_plan(cu_seqlens_host, HV):
    """(segment length in chunks, 0 when nothing is split; number of walk
    segments) that the compute calls would use for this pack and value-head
    count (host-side plan; no device work)."""
    arr, cup = _cu_host(cu_seqlens_host)
    lseg = ctypes.c_int32(0)
    nseg = ctypes.c_int64(0)
    _check(load().gdr_segment_plan(arr.shape[0] - 1, cup, int(HV), ctypes.byref(lseg), ctypes.byref(nseg)),
           "gdr_segment_plan")
    return lseg.value, nseg.value


def gdr_walk_slices(nchunks, direction):
    """Slice bounds [0, .., nchunks] of a pipelined walk over nchunks chunks:
    direction 0 the forward walk, 1 the backward (host-side plan; no device
    work)."""
    cap = nchunks + 2
    bounds = (ctypes.c_int32 * cap)()
    n = ctypes.c_int32(0)
    _check(load().gdr_walk_slices(int(nchunks), int(direction), bounds, cap, ctypes.byref(n)), "gdr_walk_slices")
    return [bounds[i] for i in range(n.value + 1)]


def kda_fwd_noalloc(q, k, v, g, beta, cu_seqlens, cu_seqlens_host, scale, out, ht=None, h0=None, stream=None):
    """KDA forward whose intermediates live in the library's fixed 64 MiB device
    array (for callers that cannot allocate; see include/gdr.h).  `out` (and
    `ht`, if wanted) must be preallocated: this wrapper allocates nothing."""
    _check_shapes("kda", q, k, v, g, beta)
    T, H, _ = q.shape
    arr, cup = _cu_host(cu_seqlens_host)
    st = load().kda_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), cup,
                                arr.shape[0] - 1, T, H, float(scale), _ptr(h0), _ptr(out), _ptr(ht), _stream(stream))
    _check(st, "kda_fwd_noalloc")
    return out, ht


def gdr_check_device():
    """Synchronize and raise GdrError if a kernel of the library timed out a
    bounded wait (or a CUDA error occurred) since the last check."""
    _check(load().gdr_check_device(), "gdr_check_device")


def gdr_inject_device_error(code: int = 1):
    """Write `code` into the device error word, as a timed-out kernel would
    (host-side fault injection for tests of the error path)."""
    _check(load().gdr_inject_device_error(int(code)), "gdr_inject_device_error")


def gdr_selftest_wait(limit_ns: int, stream=None):
    """Enqueue a kernel whose bounded wait on a barrier that nothing completes
    runs out after limit_ns; gdr_check_device() then raises GDR_DEVICE_TIMEOUT."""
    _check(load().gdr_selftest_wait(int(limit_ns), _stream(stream)), "gdr_selftest_wait")
