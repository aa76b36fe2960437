"""The C ABI without a GPU: the library loads, exports every function that
include/gdr.h declares, and its host-side logic (workspace sizing, argument
and cu_seqlens validation, the saved-buffer stamp) answers before any CUDA
call is made."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gdr():
    import gated_delta_rule_varlen_gb300 as m
    from gated_delta_rule_varlen_gb300 import build

    build.build()
    m.load()
    return m


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "gdr.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|gdr_status|int|uint64_t)\s+(\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(gdr):
    declared = _declared_functions()
    assert set(declared) == set(gdr.EXPORTED), declared
    lib = ctypes.CDLL(gdr.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(gdr):
    names = {0: "GDR_OK", 1: "GDR_INVALID_ARG", 2: "GDR_BAD_CU_SEQLENS", 3: "GDR_WORKSPACE_TOO_SMALL",
             4: "GDR_UNSUPPORTED", 5: "GDR_STALE_WORKSPACE", 6: "GDR_CUDA_ERROR", 7: "GDR_DEVICE_TIMEOUT"}
    for code, name in names.items():
        assert gdr.status_string(code) == name
    assert gdr.status_string(99) == "GDR_UNKNOWN_STATUS"


def _chunks(lengths):
    return sum((n + 63) // 64 for n in lengths)


def test_workspace_bytes_scale_with_chunks_and_heads(gdr):
    lengths = [42024, 57573, 73122, 88673]
    cu = np.cumsum([0] + lengths).astype(np.int32)
    s16, c16 = gdr.kda_workspace_bytes(int(cu[-1]), 16, cu)
    s4, c4 = gdr.kda_workspace_bytes(int(cu[-1]), 4, cu)
    NC = _chunks(lengths)
    assert NC == 4086
    # Per (chunk, head): FP16 w [64][128], Q*Gamma [64][128], Kd^T [128][64], Aqk [64][64],
    # u [64][136]; FP32 Delta [64][128], At and T [64][68] (tiles that are copied whole
    # keep their shared-memory row pitch), gamma [128]; and a 128x128 BF16 state.
    per = ((64 * 128 + 64 * 128 + 128 * 64 + 64 * 64 + 64 * 136) * 2 + (64 * 128 + 2 * 64 * 68 + 128) * 4
           + 128 * 128 * 2)
    assert s16 >= NC * 16 * per and s16 < NC * 16 * per + 1 << 20
    assert s4 >= NC * 4 * per and s4 < s16
    assert 0 < c16
    sg, cg = gdr.gdn_workspace_bytes(1000, 2, 6, [0, 500, 1000])
    sk, ck = gdr.gdn_workspace_bytes(1000, 6, 6, [0, 500, 1000])
    assert sg == sk and cg > ck  # grouped heads add per-value-head dq/dk partials


def test_workspace_validation(gdr):
    with pytest.raises(ValueError):
        gdr.kda_workspace_bytes(10, 2, [0, 5, 11])  # cu[N] != T
    with pytest.raises(ValueError):
        gdr.kda_workspace_bytes(10, 2, [0, 6, 5, 10])  # decreasing
    with pytest.raises(ValueError):
        gdr.kda_workspace_bytes(10, 2, [1, 10])  # cu[0] != 0
    with pytest.raises(ValueError):
        gdr.gdn_workspace_bytes(10, 4, 6, [0, 10])  # HV % Hqk != 0
    assert gdr.kda_workspace_bytes(0, 2, [0])[0] > 0  # no documents: tables only
    assert gdr.kda_workspace_bytes(0, 2, [0, 0, 0])[0] > 0  # empty documents


def _fake(n=1):
    return ctypes.c_void_p(0x10000 * n)  # never dereferenced: every call below fails host validation


def test_forward_host_validation_before_any_cuda_call(gdr):
    lib = gdr.load()
    cu = np.array([0, 5, 11], dtype=np.int32)
    cup = cu.ctypes.data_as(gdr.PI32)
    p = _fake()
    # cu[N] != T
    st = lib.kda_fwd(p, p, p, p, p, p, cup, 2, 10, 1, 1.0, 0, None, p, None, p, 1 << 40, 1, None, 0, None)
    assert st == gdr.GDR_BAD_CU_SEQLENS
    # workspace too small
    st = lib.kda_fwd(p, p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, p, None, _fake(256), 1024, 1, None, 0, None)
    assert st == gdr.GDR_WORKSPACE_TOO_SMALL
    # misaligned workspace
    st = lib.kda_fwd(p, p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, p, None, ctypes.c_void_p(0x10010), 1 << 40, 1,
                     None, 0, None)
    assert st == gdr.GDR_INVALID_ARG
    # null input
    st = lib.kda_fwd(None, p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, p, None, p, 1 << 40, 1, None, 0, None)
    assert st == gdr.GDR_INVALID_ARG
    # save_for_bwd without a saved buffer
    st = lib.kda_fwd(p, p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, p, None, None, 0, 1, p, 1 << 40, None)
    assert st == gdr.GDR_INVALID_ARG
    # q not on a 16-byte boundary (its rows are copied in 16-byte pieces)
    st = lib.kda_fwd(ctypes.c_void_p(0x10008), p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, p, None, p, 1 << 40, 1,
                     None, 0, None)
    assert st == gdr.GDR_INVALID_ARG
    # out not on a 4-byte boundary
    st = lib.kda_fwd(p, p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, ctypes.c_void_p(0x10002), None, p, 1 << 40, 1,
                     None, 0, None)
    assert st == gdr.GDR_INVALID_ARG
    # GDN: HV not a multiple of Hqk
    st = lib.gdn_fwd(p, p, p, p, p, p, cup, 2, 11, 4, 6, 1.0, 0, None, p, None, p, 1 << 40, 1, None, 0, None)
    assert st == gdr.GDR_INVALID_ARG
    # No documents: nothing to do.
    z = np.array([0], dtype=np.int32)
    st = lib.kda_fwd(None, None, None, None, None, None, z.ctypes.data_as(gdr.PI32), 0, 0, 1, 1.0, 0, None, None, None,
                     None, 0, 0, None, 0, None)
    assert st == gdr.GDR_OK


def test_backward_host_validation_before_any_cuda_call(gdr):
    # Every call here is rejected on the host before any work reaches the
    # device (no copy, no launch), so the fake pointers are never handed to a
    # GPU on any machine.  (A saved buffer that passes these checks goes on to
    # the device-side header check, which the GPU tests cover with real
    # buffers.)
    lib = gdr.load()
    cu = np.array([0, 5, 11], dtype=np.int32)
    cup = cu.ctypes.data_as(gdr.PI32)
    p = _fake()
    big = 1 << 40
    # cu[N] != T
    st = lib.kda_bwd(p, p, p, p, p, p, cup, 2, 10, 1, 1.0, 0, None, p, None, _fake(512), big, p, p, p, p, p, None,
                     _fake(1024), big, None)
    assert st == gdr.GDR_BAD_CU_SEQLENS
    # dout not on a 16-byte boundary
    st = lib.kda_bwd(p, p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, ctypes.c_void_p(0x10004), None, _fake(512), big, p,
                     p, p, p, p, None, _fake(1024), big, None)
    assert st == gdr.GDR_INVALID_ARG
    # misaligned scratch
    st = lib.kda_bwd(p, p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, p, None, _fake(512), big, p, p, p, p, p, None,
                     ctypes.c_void_p(0x10010), big, None)
    assert st == gdr.GDR_INVALID_ARG
    # null saved buffer
    st = lib.gdn_bwd(p, p, p, p, p, p, cup, 2, 11, 1, 3, 1.0, 0, None, p, None, None, big, p, p, p, p, p, None,
                     _fake(1024), big, None)
    assert st == gdr.GDR_INVALID_ARG
    # GDN: HV not a multiple of Hqk
    st = lib.gdn_bwd(p, p, p, p, p, p, cup, 2, 11, 4, 6, 1.0, 0, None, p, None, _fake(512), big, p, p, p, p, p, None,
                     _fake(1024), big, None)
    assert st == gdr.GDR_INVALID_ARG
    # Too-small saved buffer or scratch (reported before the stamp and the device).
    st = lib.kda_bwd(p, p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, p, None, _fake(512), 256, p, p, p, p, p, None,
                     _fake(1024), big, None)
    assert st == gdr.GDR_WORKSPACE_TOO_SMALL
    st = lib.kda_bwd(p, p, p, p, p, p, cup, 2, 11, 1, 1.0, 0, None, p, None, _fake(512), big, p, p, p, p, p, None,
                     _fake(1024), 256, None)
    assert st == gdr.GDR_WORKSPACE_TOO_SMALL


def test_binding_fails_loudly_without_library(tmp_path):
    import gated_delta_rule_varlen_gb300 as m
    saved = m._lib
    try:
        m._lib = None
        with pytest.raises(RuntimeError):
            m.load(str(tmp_path / "missing.so"))
    finally:
        m._lib = saved


def test_diagnostics_validate_arguments_before_any_cuda_call(gdr):
    lib = gdr.load()
    assert lib.gdr_inject_device_error(0) == gdr.GDR_INVALID_ARG
    assert lib.gdr_inject_device_error(-3) == gdr.GDR_INVALID_ARG
    assert lib.gdr_selftest_wait(0, None) == gdr.GDR_INVALID_ARG
    assert lib.gdr_selftest_wait(100000001, None) == gdr.GDR_INVALID_ARG


def test_binding_rejects_mismatched_shapes_before_any_device_work(gdr):
    # The C ABI receives pointers only; the binding checks the shapes it derives sizes from.
    import torch
    T = 10
    q = torch.zeros(T, 2, 128, dtype=torch.bfloat16)
    v = torch.zeros(T, 2, 128, dtype=torch.bfloat16)
    g = torch.zeros(T, 2, 128)
    beta = torch.zeros(T, 2, dtype=torch.bfloat16)
    cu = [0, T]
    with pytest.raises(ValueError):  # KDA needs as many q/k heads as v heads
        gdr.kda_fwd(q[:, :1], q[:, :1], v, g, beta, None, cu, 1.0)
    with pytest.raises(ValueError):  # KDA gate is per channel
        gdr.kda_fwd(q, q, v, g[:, :, 0], beta, None, cu, 1.0)
    with pytest.raises(ValueError):  # GDN gate is per head
        gdr.gdn_fwd(q, q, v, g, beta.float(), None, cu, 1.0)
    with pytest.raises(ValueError):  # dout shaped like v
        gdr.kda_bwd(q, q, v, g, beta, None, cu, 1.0, v[:, :1], None)
    with pytest.raises(ValueError):  # head dim 128 only
        gdr.kda_fwd(q[..., :64], q[..., :64], v[..., :64], g[..., :64], beta, None, cu, 1.0)
