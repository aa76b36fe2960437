"""The no-allocation KDA forward (kda_fwd_noalloc), called through the C ABI.

Some callers cannot allocate device memory when they call the library: code
under CUDA stream capture in global mode, engines whose framework owns all
device memory, real-time paths that must not hit the allocator.  For them
kda_fwd_noalloc keeps the forward's intermediates in a fixed 64 MiB device
array inside the library.  This test checks it against the regular kda_fwd on
the same inputs, on two calls in a row (the array keeps the first call's
contents when the second starts), and that a problem too large for the array
is rejected before anything runs.  This file is named to be collected last.
"""
import ctypes

import pytest
import torch

import synth
from gpu_util import SCALE, TOL, assert_within, compare, f64, rel, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import gated_delta_rule_varlen_gb300 as gdr
    return gdr


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(gdr, x, cu_d, cu, H, out, ht, h0=None):
    import numpy as np
    cuh = np.asarray(cu, dtype=np.int32)
    st = gdr.load().kda_fwd_noalloc(
        _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["g"]), _p(x["beta"]), _p(cu_d), cuh.ctypes.data_as(gdr.PI32),
        len(cu) - 1, cu[-1], H, SCALE, _p(h0), _p(out), _p(ht),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_forward_matches_kda_fwd_twice(lib):
    gdr = lib
    cases = [([1000, 37, 513], 2, 0), ([64, 700, 1], 2, 1)]  # second call differs in shape and contents
    outs = []
    for lengths, H, seed in cases:
        T = sum(lengths)
        cu = synth.cu_from_lengths(lengths)
        x = {k: v.cuda() for k, v in synth.make_inputs("kda", T, H, H, 128, seed=seed).items()}
        cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
        h0 = synth.make_states(len(lengths), H, 128, seed=seed + 3, scale=0.05).cuda()
        ref_out, ref_ht, _ = gdr.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_d, cu, SCALE, h0=h0,
                                         save_for_bwd=False)
        out = torch.full_like(ref_out, float("nan"))
        ht = torch.full_like(ref_ht, float("nan"))
        st = _noalloc(gdr, x, cu_d, cu, H, out, ht, h0=h0)
        assert st == gdr.GDR_OK, gdr.status_string(st)
        torch.cuda.synchronize()
        e_out, e_ht = rel(f64(out), f64(ref_out)), rel(f64(ht), f64(ref_ht))
        assert e_out <= TOL["out"] and e_ht <= TOL["ht"], (e_out, e_ht)
        outs.append((out, ref_out))
    for out, ref in outs:
        assert torch.isfinite(out).all()


def test_noalloc_forward_multi_group_matches_oracle(lib):
    # Three documents of 64 chunks each run as document groups of their own and the short
    # fourth as one more: four groups forked onto the library's internal streams, with the
    # intermediates in the fixed array (about 50 MB of it).  Checked against the FP64 oracle,
    # twice in a row.
    gdr = lib
    lengths, H = [4096, 4096, 4096, 100], 1
    T = sum(lengths)
    cu = synth.cu_from_lengths(lengths)
    assert len(gdr.gdr_doc_groups(cu)) == 4
    saved_bytes, _ = gdr.kda_workspace_bytes(T, H, cu)
    assert saved_bytes <= 64 << 20
    xh = synth.make_inputs("kda", T, H, H, 128, seed=21)
    h0h = synth.make_states(len(lengths), H, 128, seed=22, scale=0.05)
    x = {k: v.cuda() for k, v in xh.items()}
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    ref = run_oracle(xh, cu, h0=h0h, backward=False)
    for _ in range(2):
        out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        ht = torch.full((len(lengths), H, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc(gdr, x, cu_d, cu, H, out, ht, h0=h0h.cuda())
        assert st == gdr.GDR_OK, gdr.status_string(st)
        torch.cuda.synchronize()
        gdr.gdr_check_device()
        print("noalloc multi-group", assert_within(compare({"out": out, "ht": ht}, ref)))


def test_noalloc_rejects_problem_beyond_the_fixed_array(lib):
    gdr = lib
    lengths = [16384, 16384]  # 512 chunks x 4 heads: far above 64 MiB of intermediates
    T, H = sum(lengths), 4
    cu = synth.cu_from_lengths(lengths)
    saved_bytes, _ = gdr.kda_workspace_bytes(T, H, cu)
    assert saved_bytes > 64 << 20
    x = {k: v.cuda() for k, v in synth.make_inputs("kda", T, H, H, 128, seed=5).items()}
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out = torch.empty((T, H, 128), dtype=torch.bfloat16, device="cuda")
    st = _noalloc(gdr, x, cu_d, cu, H, out, None)
    assert st == gdr.GDR_WORKSPACE_TOO_SMALL
