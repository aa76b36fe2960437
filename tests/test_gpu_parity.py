"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle on
the same seeded inputs.  Small cases compare every element; the full-size
workloads compare sampled (document, head) chains, which the oracle computes
independently of the rest of the pack.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import SCALE, TOL, assert_within, compare, err_stats, f64, rel, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import gated_delta_rule_varlen_gb300 as gdr
    gdr.load()


def _case(variant, lengths, Hqk, HV, seed=0, h0=False, dht=False, glow=-5.0, ghigh=0.0):
    T = sum(lengths)
    cu = synth.cu_from_lengths(lengths)
    x = synth.make_inputs(variant, T, Hqk, HV, 128, seed=seed, gate_low=glow, gate_high=ghigh)
    h0t = synth.make_states(len(lengths), HV, 128, seed=seed + 11, scale=0.05) if h0 else None
    dhtt = synth.make_states(len(lengths), HV, 128, seed=seed + 12, scale=0.05) if dht else None
    return x, cu, h0t, dhtt


def _check(variant, lengths, Hqk, HV, **kw):
    x, cu, h0, dht = _case(variant, lengths, Hqk, HV, **kw)
    gpu = run_gpu(variant, x, cu, h0=h0, dht=dht, want_dh0=h0 is not None)
    ref = run_oracle(x, cu, h0=h0, dht=dht)
    errs = compare(gpu, ref)
    print(variant, lengths, assert_within(errs))
    return gpu, ref


def test_kda_tiny_config():
    # One document of 512 tokens, H = 1, seed 0.
    _check("kda", [512], 1, 1)


def test_kda_ragged_edges_with_states():
    _check("kda", [1, 63, 64, 65, 0, 127, 128, 129, 200], 2, 2, seed=1, h0=True, dht=True)


def test_gdn_grouped_ragged_with_states():
    _check("gdn", [5, 64, 130, 0, 71], 2, 6, seed=2, h0=True, dht=True)


def test_gdn_production_heads_small_pack():
    _check("gdn", [300, 211], 16, 48, seed=3)


def test_gdn_ungrouped_heads_ragged():
    # One value head per Q/K head (no grouping): the prep's per-group loop runs once.
    _check("gdn", [1, 63, 64, 65, 0, 129], 2, 2, seed=23, h0=True, dht=True)


def test_gdn_eight_value_heads_per_qk_head():
    # Eight value heads share each Q/K head's Gram; gate and v tiles rotate through the buffers.
    _check("gdn", [100, 64, 77], 1, 8, seed=24, h0=True, dht=True)


def test_kda_large_values_within_the_fp16_operand_range():
    # The forward walk multiplies FP16 copies of the state and of Delta, which
    # scale with the values v: v 300 times larger than the workloads' (entries
    # up to ~1e3, state entries in the thousands) stays well inside FP16's range.
    x, cu, h0, dht = _case("kda", [700, 129], 2, 2, seed=25, glow=-0.05, h0=True, dht=True)
    x["v"] = (x["v"].float() * 300.0).to(torch.bfloat16)
    h0 = h0 * 300.0
    gpu = run_gpu("kda", x, cu, h0=h0, dht=dht, want_dh0=True)
    ref = run_oracle(x, cu, h0=h0, dht=dht)
    print("large v", assert_within(compare(gpu, ref)))


def test_kda_mild_gates_long_document():
    # Gates near zero keep the state alive across all 64 chunks.
    _check("kda", [4096], 1, 1, seed=4, glow=-0.05, h0=True, dht=True)


def test_gdn_mild_gates_long_document():
    _check("gdn", [4096], 1, 2, seed=5, glow=-0.05, h0=True)


def test_kda_zero_gate():
    _check("kda", [1000], 1, 1, seed=6, glow=0.0, ghigh=0.0)


def test_kda_strong_gates_lower_bound():
    # Gates down to -10 (the library's stated lower bound).
    _check("kda", [300], 1, 1, seed=7, glow=-10.0)


def test_packed_equals_per_document_bitwise():
    lengths = [70, 1, 130, 64]
    x, cu, h0, dht = _case("kda", lengths, 2, 2, seed=8, h0=True, dht=True)
    whole = run_gpu("kda", x, cu, h0=h0, dht=dht, want_dh0=True)
    for n in range(len(lengths)):
        s, e = cu[n], cu[n + 1]
        xs = {k: v[s:e] for k, v in x.items()}
        one = run_gpu("kda", xs, [0, e - s], h0=h0[n:n + 1], dht=dht[n:n + 1], want_dh0=True)
        for name in ("out", "dq", "dk", "dv", "dg", "dbeta"):
            assert torch.equal(whole[name][s:e], one[name]), name
        assert torch.equal(whole["ht"][n], one["ht"][0])
        assert torch.equal(whole["dh0"][n], one["dh0"][0])


def test_kda_document_groups_on_their_own_streams():
    # Three documents of at least 64 chunks run as groups of their own, the rest as one more
    # (four streams in the forward and the backward); every element against the oracle.
    import gated_delta_rule_varlen_gb300 as gdr
    lengths = [4200, 130, 4096, 0, 4500, 64]
    assert len(gdr.gdr_doc_groups(synth.cu_from_lengths(lengths))) == 4
    _check("kda", lengths, 2, 2, seed=13, h0=True, dht=True)


def test_gdn_document_groups_on_their_own_streams():
    import gated_delta_rule_varlen_gb300 as gdr
    lengths = [100, 4160, 5000]
    assert len(gdr.gdr_doc_groups(synth.cu_from_lengths(lengths))) == 3
    _check("gdn", lengths, 1, 2, seed=14, h0=True, dht=True)


def test_document_groups_with_an_empty_last_group():
    # Three long documents stand alone; the remaining group holds only an empty document, whose
    # final state is its initial state and whose dh0 is its dht.
    import gated_delta_rule_varlen_gb300 as gdr
    lengths = [4200, 4096, 0, 4500]
    groups = gdr.gdr_doc_groups(synth.cu_from_lengths(lengths))
    assert len(groups) == 4 and groups[3][2] == groups[3][3]
    gpu, _ = _check("kda", lengths, 2, 2, seed=18, h0=True, dht=True)
    x, cu, h0, dht = _case("kda", lengths, 2, 2, seed=18, h0=True, dht=True)
    assert torch.equal(gpu["ht"][2].cpu(), h0[2])
    assert torch.equal(gpu["dh0"][2].cpu(), dht[2])


def test_more_documents_than_the_ranking_limit():
    # Above 4096 documents the plan keeps the given order; the long first document is still a
    # group of its own.
    import gated_delta_rule_varlen_gb300 as gdr
    lengths = [10000] + [10] * 4097
    assert len(gdr.gdr_doc_groups(synth.cu_from_lengths(lengths))) == 2
    _check("kda", lengths, 1, 1, seed=17)


def test_grouped_pack_equals_per_document_bitwise():
    lengths = [4200, 70, 4096, 4500]
    x, cu, h0, dht = _case("kda", lengths, 2, 2, seed=15, h0=True, dht=True)
    whole = run_gpu("kda", x, cu, h0=h0, dht=dht, want_dh0=True)
    for n in range(len(lengths)):
        s, e = cu[n], cu[n + 1]
        xs = {k: v[s:e] for k, v in x.items()}
        one = run_gpu("kda", xs, [0, e - s], h0=h0[n:n + 1], dht=dht[n:n + 1], want_dh0=True)
        for name in ("out", "dq", "dk", "dv", "dg", "dbeta"):
            assert torch.equal(whole[name][s:e], one[name]), name
        assert torch.equal(whole["ht"][n], one["ht"][0])
        assert torch.equal(whole["dh0"][n], one["dh0"][0])


def test_repeat_is_bitwise_deterministic():
    x, cu, h0, dht = _case("gdn", [200, 333], 2, 6, seed=9)
    a = run_gpu("gdn", x, cu)
    b = run_gpu("gdn", x, cu)
    for name in ("out", "ht", "dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(a[name], b[name]), name


def test_empty_documents_pass_state_through():
    x, cu, h0, dht = _case("kda", [0, 0], 1, 1, seed=10, h0=True, dht=True)
    gpu = run_gpu("kda", x, cu, h0=h0, dht=dht, want_dh0=True)
    assert torch.equal(gpu["ht"].cpu(), h0)
    assert torch.equal(gpu["dh0"].cpu(), dht)


def test_workspace_errors_on_gpu():
    import gated_delta_rule_varlen_gb300 as gdr
    x, cu, _, _ = _case("kda", [100], 1, 1, seed=11)
    xd = {k: v.cuda() for k, v in x.items()}
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out, ht, saved = gdr.kda_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE)
    # A saved buffer stamped for another pack is rejected.
    with pytest.raises(gdr.GdrError) as ei:
        cu2 = [0, 50, 100]
        gdr.kda_bwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], torch.tensor(cu2, dtype=torch.int32,
                    device="cuda"), cu2, SCALE, xd["dout"], saved)
    assert ei.value.status == gdr.GDR_STALE_WORKSPACE
    # Too-small scratch.
    with pytest.raises(ValueError):
        gdr.kda_bwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE, xd["dout"], saved,
                    scratch=torch.empty(1024, dtype=torch.uint8, device="cuda"))


def _kda_small(lengths, seed):
    x, cu, _, _ = _case("kda", lengths, 2, 2, seed=seed)
    xd = {k: v.cuda() for k, v in x.items()}
    return xd, torch.tensor(cu, dtype=torch.int32, device="cuda"), cu


def test_saved_buffer_copied_to_another_address_is_accepted():
    # The saved buffer's header travels with it: a copy at another address,
    # unknown to the host registry, gives the same gradients.
    import gated_delta_rule_varlen_gb300 as gdr
    gdr.gdr_check_device()
    xd, cu_d, cu = _kda_small([300, 77], 13)
    args = (xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE)
    _, _, saved = gdr.kda_fwd(*args)
    a = gdr.kda_bwd(*args, xd["dout"], saved)
    b = gdr.kda_bwd(*args, xd["dout"], saved.clone())
    gdr.gdr_check_device()
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(a[name], b[name]), name


def test_saved_buffer_overwritten_or_clobbered_is_reported():
    import gated_delta_rule_varlen_gb300 as gdr
    gdr.gdr_check_device()
    xd, cu_d, cu = _kda_small([300, 77], 14)
    args = (xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE)
    _, _, s1 = gdr.kda_fwd(*args)
    _, _, s2 = gdr.kda_fwd(*args)
    # Another forward's saved buffer copied over a registered one: same
    # problem, but the header names another forward than the one the host
    # registry recorded for this address.
    s1.copy_(s2)
    gdr.kda_bwd(*args, xd["dout"], s1)
    with pytest.raises(gdr.GdrError) as ei:
        gdr.gdr_check_device()
    assert ei.value.status == gdr.GDR_STALE_WORKSPACE
    gdr.gdr_check_device()  # the report cleared the word
    # A copy (unregistered) whose magic word was overwritten.
    c = s2.clone()
    c[:8] = 0
    gdr.kda_bwd(*args, xd["dout"], c)
    with pytest.raises(gdr.GdrError) as ei:
        gdr.gdr_check_device()
    assert ei.value.status == gdr.GDR_STALE_WORKSPACE
    # The registered, untouched buffer still works, and the context is usable.
    ref = run_gpu("kda", {k: v.cpu() for k, v in xd.items()}, cu)
    good = gdr.kda_bwd(*args, xd["dout"], s2)
    gdr.gdr_check_device()
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(good[name], ref[name]), name


def test_ckpt_sequence_matches_plain_backward():
    # ckpt = forward (no save), forward (save), backward: same results as forward + backward.
    import gated_delta_rule_varlen_gb300 as gdr
    x, cu, _, _ = _case("kda", [300, 77], 2, 2, seed=12)
    xd = {k: v.cuda() for k, v in x.items()}
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    a = run_gpu("kda", x, cu)
    o1, _, _ = gdr.kda_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE, save_for_bwd=False)
    o2, _, saved = gdr.kda_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE)
    gr = gdr.kda_bwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE, xd["dout"], saved)
    assert torch.equal(o1, a["out"]) and torch.equal(o2, a["out"])
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(gr[name], a[name]), name


# ---------------------------------------------------------------------------
# Full-size workloads: sampled chains.
# ---------------------------------------------------------------------------
def _full_case(name, seed=0):
    wl = synth.workload(name)
    x = synth.make_inputs(wl.variant, wl.T, wl.Hqk, wl.HV, 128, seed=seed, device="cuda")
    return wl, x


def _sample_check(wl, x, gpu, samples):
    """samples: list of (doc, qk_head).  The oracle runs the chains of that
    document for every value head of the Q/K head (GDN: the whole group)."""
    from concurrent.futures import ThreadPoolExecutor
    cu = wl.cu_seqlens
    G = wl.HV // wl.Hqk

    def one(sample):
        n, hq = sample
        s, e = cu[n], cu[n + 1]
        hv = list(range(hq * G, hq * G + G))
        xs = {
            "q": x["q"][s:e, hq:hq + 1].cpu(), "k": x["k"][s:e, hq:hq + 1].cpu(),
            "v": x["v"][s:e, hv].cpu(), "g": x["g"][s:e, hv].cpu(), "beta": x["beta"][s:e, hv].cpu(),
            "dout": x["dout"][s:e, hv].cpu(),
        }
        ref = run_oracle(xs, [0, e - s])
        got = {
            "out": f64(gpu["out"][s:e, hv]), "ht": f64(gpu["ht"][n, hv]), "dq": f64(gpu["dq"][s:e, hq:hq + 1]),
            "dk": f64(gpu["dk"][s:e, hq:hq + 1]), "dv": f64(gpu["dv"][s:e, hv]), "dg": f64(gpu["dg"][s:e, hv]),
            "dbeta": f64(gpu["dbeta"][s:e, hv]),
        }
        return sample, {k: err_stats(got[k], ref[k]) for k in got}

    with ThreadPoolExecutor(max_workers=len(samples)) as ex:
        results = list(ex.map(one, samples))
    for sample, errs in results:
        print(wl.name, sample, assert_within(errs))


def _every_group_samples(wl, heads):
    """One (document, Q/K head) sample per document group of the pack: the
    documents in longest-first order take the given heads in turn, so the
    longest document (the longest chain) is always sampled, and every group
    (each of the three longest documents with >= 64 chunks is a group of its
    own; the rest form one more) is covered.  For packs of more documents
    than heads the shortest document is added as well."""
    import gated_delta_rule_varlen_gb300 as gdr
    order = sorted(range(len(wl.lengths)), key=lambda n: (-wl.lengths[n], n))
    rank_of = {n: r for r, n in enumerate(order)}
    groups = gdr.gdr_doc_groups(wl.cu_seqlens)
    picks = []
    for (r0, r1, _, _) in groups:
        picks.append(order[r0])  # the group's longest document
    shortest = order[-1]
    if shortest not in picks:
        picks.append(shortest)
    assert picks[0] == order[0] and all(any(r0 <= rank_of[n] < r1 for n in picks) for r0, r1, _, _ in groups)
    return [(n, heads[i % len(heads)]) for i, n in enumerate(picks)]


@pytest.mark.slow
@pytest.mark.parametrize("name,heads", [
    ("kda_pack_h16", [3, 11, 0, 15]),
    ("kda_pack_h4", [0, 1, 2, 3]),
    ("kda_pack_h64", [63, 17, 40, 5]),
])
def test_fullsize_kda_sampled_chains(name, heads):
    wl, x = _full_case(name)
    gpu = run_gpu("kda", x, wl.cu_seqlens)
    for k in ("out", "dq", "dk", "dv", "dg", "dbeta"):
        assert torch.isfinite(gpu[k]).all(), k
    _sample_check(wl, x, gpu, _every_group_samples(wl, heads))


@pytest.mark.slow
@pytest.mark.parametrize("name,heads", [
    ("gdn_p1", [7, 0, 15, 9]),
    ("gdn_1doc", [2]),
])
def test_fullsize_gdn_sampled_chains(name, heads):
    wl, x = _full_case(name)
    gpu = run_gpu("gdn", x, wl.cu_seqlens)
    for k in ("out", "dq", "dk", "dv", "dg", "dbeta"):
        assert torch.isfinite(gpu[k]).all(), k
    samples = _every_group_samples(wl, heads)
    assert int(np.argmax(wl.lengths)) == samples[0][0] and int(np.argmin(wl.lengths)) in [n for n, _ in samples]
    _sample_check(wl, x, gpu, samples)


@pytest.mark.slow
def test_fullsize_ckpt_sequence_matches_plain_backward():
    # ckpt at the H = 16 pack: forward (no save), forward (save), backward gives the plain
    # forward + backward results bit for bit (the plain results are oracle-checked above).
    import gated_delta_rule_varlen_gb300 as gdr
    wl, x = _full_case("kda_pack_h16")
    cu = wl.cu_seqlens
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o0, h0_, saved = gdr.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_d, cu, SCALE)
    g0 = gdr.kda_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_d, cu, SCALE, x["dout"], saved)
    del saved
    o1, _, _ = gdr.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_d, cu, SCALE, save_for_bwd=False)
    o2, _, saved = gdr.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_d, cu, SCALE)
    g1 = gdr.kda_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu_d, cu, SCALE, x["dout"], saved)
    torch.cuda.synchronize()
    gdr.gdr_check_device()
    assert torch.equal(o1, o0) and torch.equal(o2, o0)
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(g1[name], g0[name]), name


def test_graph_capture_of_grouped_fwd_bwd_replays_bitwise():
    # The document groups fork onto internal streams; a captured fwd + bwd must replay to the
    # eager results, bit for bit.
    import gated_delta_rule_varlen_gb300 as gdr
    lengths = [4200, 130, 4096, 4500]
    x, cu, _, _ = _case("kda", lengths, 1, 1, seed=16)
    xd = {k: v.cuda() for k, v in x.items()}
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")

    def step():
        out, ht, saved = gdr.kda_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE)
        grads = gdr.kda_bwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE, xd["dout"], saved)
        return out, ht, grads

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        eager = step()  # also creates the library's internal streams before the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = step()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(cap[0], eager[0]) and torch.equal(cap[1], eager[1])
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(cap[2][name], eager[2][name]), name


# ---------------------------------------------------------------------------
# Segment-parallel walks: documents split into segments walked in parallel
# (summary walks, a merge of the segment start states, then every segment's
# walk).  Forced to short segments so that small cases cover one, two (no
# merge) and many segments per document.
# ---------------------------------------------------------------------------
@pytest.fixture
def segments():
    import gated_delta_rule_varlen_gb300 as gdr

    def force(chunks):
        gdr.gdr_set_segment_chunks(chunks)

    yield force
    gdr.gdr_set_segment_chunks(0)


def test_kda_segments_mild_gates_long_document(segments):
    # 64 chunks in segments of 8: 8 segments, 6 merged; mild gates keep the state alive across
    # all of them, so a wrong segment map or start state shows in out, ht and every gradient.
    segments(8)
    _check("kda", [4096], 1, 1, seed=4, glow=-0.05, h0=True, dht=True)


def test_kda_segments_zero_gate(segments):
    segments(3)
    _check("kda", [1000], 1, 1, seed=6, glow=0.0, ghigh=0.0, h0=True, dht=True)


def test_gdn_segments_grouped_mild_gates(segments):
    segments(5)
    _check("gdn", [4096, 700], 1, 3, seed=5, glow=-0.05, h0=True, dht=True)


def test_kda_segments_ragged_pack(segments):
    # Segments of 5 chunks: documents of 1 (16 chunks: 4 segments), 2 (10 chunks, no merge),
    # 1 segment (5 chunks and 1 token), an empty document, and a long one (13 segments).
    segments(5)
    _check("kda", [1000, 640, 300, 1, 0, 4096], 2, 2, seed=19, glow=-0.2, h0=True, dht=True)


def test_segments_packed_equals_per_document_bitwise(segments):
    segments(4)
    lengths = [1500, 64, 700]
    x, cu, h0, dht = _case("kda", lengths, 2, 2, seed=20, h0=True, dht=True, glow=-0.3)
    whole = run_gpu("kda", x, cu, h0=h0, dht=dht, want_dh0=True)
    for n in range(len(lengths)):
        s, e = cu[n], cu[n + 1]
        xs = {k: v[s:e] for k, v in x.items()}
        one = run_gpu("kda", xs, [0, e - s], h0=h0[n:n + 1], dht=dht[n:n + 1], want_dh0=True)
        for name in ("out", "dq", "dk", "dv", "dg", "dbeta"):
            assert torch.equal(whole[name][s:e], one[name]), name
        assert torch.equal(whole["ht"][n], one["ht"][0])
        assert torch.equal(whole["dh0"][n], one["dh0"][0])


def test_segments_ckpt_matches_plain(segments):
    import gated_delta_rule_varlen_gb300 as gdr
    segments(6)
    x, cu, _, _ = _case("kda", [3000, 500], 2, 2, seed=12)
    xd = {k: v.cuda() for k, v in x.items()}
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    a = run_gpu("kda", x, cu)
    o1, _, _ = gdr.kda_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE, save_for_bwd=False)
    o2, _, saved = gdr.kda_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE)
    gr = gdr.kda_bwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE, xd["dout"], saved)
    assert torch.equal(o1, a["out"]) and torch.equal(o2, a["out"])
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(gr[name], a[name]), name


# ---------------------------------------------------------------------------
# In-kernel q/k L2 normalization (qk_l2norm): raw q, k with row norms from
# about 0.25 to 4 x sqrt(128); the oracle normalizes in FP64.
# ---------------------------------------------------------------------------
def _check_l2(variant, lengths, Hqk, HV, seed, glow=-5.0, states=True):
    T = sum(lengths)
    cu = synth.cu_from_lengths(lengths)
    x = synth.make_inputs(variant, T, Hqk, HV, 128, seed=seed, gate_low=glow, normalize_qk=False)
    h0 = synth.make_states(len(lengths), HV, 128, seed=seed + 11, scale=0.05) if states else None
    dht = synth.make_states(len(lengths), HV, 128, seed=seed + 12, scale=0.05) if states else None
    gpu = run_gpu(variant, x, cu, h0=h0, dht=dht, want_dh0=states, l2=True)
    ref = run_oracle(x, cu, h0=h0, dht=dht, l2=True)
    print(variant, "l2", lengths, assert_within(compare(gpu, ref)))
    return gpu, x


def test_kda_qk_l2norm():
    gpu, x = _check_l2("kda", [300, 77, 0, 129], 2, 2, seed=40)
    # The gradient with respect to a vector that is normalized has no component along it.
    dot = (gpu["dq"].double() * x["q"].cuda().double()).sum(-1).abs().max().item()
    assert dot < 2e-2 * gpu["dq"].double().norm(dim=-1).max().item()


def test_gdn_qk_l2norm_grouped():
    _check_l2("gdn", [5, 64, 130, 71], 2, 6, seed=41)


def test_kda_qk_l2norm_mild_gates_long_document():
    _check_l2("kda", [4096], 1, 1, seed=42, glow=-0.05)


# ---------------------------------------------------------------------------
# Pipelined walks: a group's one long document walked slice by slice (forced
# short slices here), the prep (forward) or the gradient kernels (backward)
# of each slice running beside the next slice's walk.
# ---------------------------------------------------------------------------
@pytest.fixture
def slices():
    import gated_delta_rule_varlen_gb300 as gdr

    def force(chunks):
        gdr.gdr_set_slice_chunks(chunks)

    yield force
    gdr.gdr_set_slice_chunks(0)


def test_kda_pipelined_walks_mild_gates_long_document(slices):
    # 64 chunks in slices of 16 (also one of 10, which rounds to an even 10): the state and
    # the adjoint cross every slice boundary through the carry buffers.
    for sl in (16, 10):
        slices(sl)
        _check("kda", [4096], 2, 2, seed=31, glow=-0.05, h0=True, dht=True)


def test_gdn_pipelined_walks_grouped_with_a_rest_group(slices):
    # A pipelined 64-chunk document beside a group of short ones (walked whole).
    slices(12)
    _check("gdn", [4096, 700, 65], 1, 3, seed=32, glow=-0.05, h0=True, dht=True)


def test_pipelined_walks_equal_whole_walks_bitwise(slices):
    # Slicing only reorders launches: every output is bit for bit the whole walk's.
    for variant, hqk, hv in (("kda", 2, 2), ("gdn", 1, 3)):
        x, cu, h0, dht = _case(variant, [4096, 300], hqk, hv, seed=33, h0=True, dht=True)
        slices(0)
        a = run_gpu(variant, x, cu, h0=h0, dht=dht, want_dh0=True)
        slices(8)
        b = run_gpu(variant, x, cu, h0=h0, dht=dht, want_dh0=True)
        for name in a:
            if a[name] is not None:
                assert torch.equal(a[name], b[name]), (variant, name)


def test_pipelined_walks_uneven_slices_equal_whole_walks_bitwise(slices):
    # Documents of 67 chunks (odd: the last slice takes the extra chunk) and 65 chunks (with
    # slices of 64 the forward's end slices of 32 do not fit, and it is cut into slices of 64
    # and 1), both ragged in their last chunk, against their whole walks.
    for variant, hqk, hv in (("kda", 2, 2), ("gdn", 1, 3)):
        x, cu, h0, dht = _case(variant, [4250, 4100], hqk, hv, seed=36, h0=True, dht=True)
        slices(0)
        a = run_gpu(variant, x, cu, h0=h0, dht=dht, want_dh0=True)
        for sl in (8, 64):
            slices(sl)
            b = run_gpu(variant, x, cu, h0=h0, dht=dht, want_dh0=True)
            for name in a:
                if a[name] is not None:
                    assert torch.equal(a[name], b[name]), (variant, sl, name)


def test_pipelined_walks_ckpt_and_l2(slices):
    # The checkpoint sequence and the in-kernel L2 norm with pipelined walks.
    import gated_delta_rule_varlen_gb300 as gdr
    slices(16)
    x, cu, _, _ = _case("kda", [4096, 77], 2, 2, seed=34, glow=-0.05)
    xd = {k: v.cuda() for k, v in x.items()}
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    a = run_gpu("kda", x, cu)
    o1, _, _ = gdr.kda_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE, save_for_bwd=False)
    o2, _, saved = gdr.kda_fwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE)
    gr = gdr.kda_bwd(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cu_d, cu, SCALE, xd["dout"], saved)
    assert torch.equal(o1, a["out"]) and torch.equal(o2, a["out"])
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(gr[name], a[name]), name
    _check_l2("kda", [4096, 77], 2, 2, seed=35)
