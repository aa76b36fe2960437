"""Pins of the FP64 oracle to facts that do not come from the oracle itself.

Each test would fail on a plausible mistake in the oracle: a dropped term, a
wrong sign, a transposed operand, a gate applied to the wrong index, a state
not reset at a document start, a wrong grouped-head mapping.

* Finite differences: every gradient (dq, dk, dv, dg, dbeta, dh0) equals the
  central difference of L = <out, dout> + <ht, dht> (KDA and grouped GDN).
* Delta-rule write: with beta = 1 and unit keys, S_t^T k_t = v_t at every
  token whatever the gates and history, so q = k gives out = scale * v.
* One token from a zero state: out = scale * beta (q.k) v, with hand-written
  gradients; dg = 0 because the gate only multiplies the zero state.
* beta = 0: the state only decays, out_t = scale (diag(exp(sum g)) h0)^T q_t.
* Orthogonal keys: the delta correction vanishes and the rule reduces to
  (decayed) causal linear attention, a masked matrix product.
* Packed == per-document (bitwise), empty documents pass h0 -> ht.
* KDA <-> GDN: a scalar gate equals a per-channel gate broadcast; grouped GDN
  equals ungrouped GDN on repeated q, k with dq, dk summed per group.
"""
import numpy as np
import pytest

import oracle


def _rand_problem(rng, lengths, Hqk, HV, D, per_channel, glow=-1.0, with_h0=True):
    T = sum(lengths)
    q = rng.standard_normal((T, Hqk, D))
    k = rng.standard_normal((T, Hqk, D))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, HV, D))
    g = rng.uniform(glow, 0.0, (T, HV, D) if per_channel else (T, HV))
    beta = rng.uniform(0.0, 1.0, (T, HV))
    N = len(lengths)
    h0 = rng.standard_normal((N, HV, D, D)) if with_h0 else None
    dout = rng.standard_normal((T, HV, D))
    dht = rng.standard_normal((N, HV, D, D))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, dout=dout, dht=dht, cu=cu)


def _loss(P, scale, l2=False, **over):
    x = dict(P)
    x.update(over)
    r = oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], scale, h0=x["h0"], qk_l2norm=l2)
    return float((r["out"] * x["dout"]).sum() + (r["ht"] * x["dht"]).sum())


def _check_fd(P, scale, eps=1e-6, tol=1e-6, l2=False):
    r = oracle.run(P["q"], P["k"], P["v"], P["g"], P["beta"], P["cu"], scale,
                   h0=P["h0"], dout=P["dout"], dht=P["dht"], qk_l2norm=l2)
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"), ("h0", "dh0")]
    for name, gname in names:
        x = P[name]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            fd[idx] = (_loss(P, scale, l2, **{name: xp}) - _loss(P, scale, l2, **{name: xm})) / (2 * eps)
        an = r[gname]
        err = np.abs(an - fd).max() / max(np.abs(fd).max(), 1e-12)
        assert err < tol, f"{gname}: finite-difference mismatch {err:.3e}"


def test_fd_gradients_kda():
    rng = np.random.default_rng(0)
    P = _rand_problem(rng, [3, 1, 5], Hqk=2, HV=2, D=4, per_channel=True)
    _check_fd(P, scale=0.7)


def test_fd_gradients_gdn_grouped():
    rng = np.random.default_rng(1)
    P = _rand_problem(rng, [4, 2], Hqk=2, HV=6, D=4, per_channel=False)
    _check_fd(P, scale=0.5)


def test_fd_gradients_with_empty_document():
    rng = np.random.default_rng(2)
    P = _rand_problem(rng, [2, 0, 3], Hqk=1, HV=1, D=4, per_channel=True)
    _check_fd(P, scale=1.0)


# The reverse pass replays each chain from square-root checkpoints taken every
# max(ceil(sqrt(L)), 16) tokens.  Documents of 40, 23 and 37 tokens hold three,
# two and three such segments, so these cases run the segment replay (which
# checkpoint a segment starts from, where it ends, the adjoint carried across
# a segment boundary) under the same independent finite-difference check.
def test_fd_gradients_kda_multi_segment_replay():
    rng = np.random.default_rng(20)
    P = _rand_problem(rng, [40, 23], Hqk=2, HV=2, D=4, per_channel=True, glow=-0.3)
    _check_fd(P, scale=0.6)


def test_fd_gradients_gdn_grouped_multi_segment_replay():
    rng = np.random.default_rng(21)
    P = _rand_problem(rng, [37], Hqk=1, HV=3, D=4, per_channel=False, glow=-0.3)
    _check_fd(P, scale=0.8)


def test_delta_rule_write_invariant():
    # beta = 1, |k| = 1, q = k  =>  out_t = scale * S_t^T k_t = scale * v_t for every t.
    rng = np.random.default_rng(3)
    for per_channel in (True, False):
        P = _rand_problem(rng, [7, 13, 1], Hqk=2, HV=2, D=8, per_channel=per_channel, glow=-3.0)
        beta = np.ones_like(P["beta"])
        r = oracle.run(P["k"], P["k"], P["v"], P["g"], beta, P["cu"], 0.3, h0=P["h0"])
        np.testing.assert_allclose(r["out"], 0.3 * P["v"], rtol=0, atol=1e-12)
    # The special case: g = 0, zero state, one token.
    k = rng.standard_normal((1, 1, 8)); k /= np.linalg.norm(k)
    v = rng.standard_normal((1, 1, 8))
    r = oracle.run(k, k, v, np.zeros((1, 1, 8)), np.ones((1, 1)), [0, 1], 1.0)
    np.testing.assert_allclose(r["ht"][0, 0].T @ k[0, 0], v[0, 0], atol=1e-14)


def test_one_token_closed_form():
    rng = np.random.default_rng(4)
    D = 8
    q, k, v, do = (rng.standard_normal((1, 1, D)) for _ in range(4))
    g = rng.uniform(-2, 0, (1, 1, D))
    b = np.array([[0.37]])
    s = 0.25
    r = oracle.run(q, k, v, g, b, [0, 1], s, dout=do)
    qk = float(q.ravel() @ k.ravel())
    vdo = float(v.ravel() @ do.ravel())
    np.testing.assert_allclose(r["out"].ravel(), s * 0.37 * qk * v.ravel(), rtol=1e-13)
    np.testing.assert_allclose(r["dq"].ravel(), s * 0.37 * vdo * k.ravel(), rtol=1e-12)
    np.testing.assert_allclose(r["dk"].ravel(), s * 0.37 * vdo * q.ravel(), rtol=1e-12)
    np.testing.assert_allclose(r["dv"].ravel(), s * 0.37 * qk * do.ravel(), rtol=1e-12)
    np.testing.assert_allclose(r["dbeta"].ravel(), [s * qk * vdo], rtol=1e-12)
    np.testing.assert_allclose(r["dg"], 0.0, atol=1e-15)
    np.testing.assert_allclose(r["ht"][0, 0], 0.37 * np.outer(k.ravel(), v.ravel()), rtol=1e-13)


def test_beta_zero_pure_decay():
    rng = np.random.default_rng(5)
    T, D = 9, 8
    q = rng.standard_normal((T, 1, D)); k = rng.standard_normal((T, 1, D)); v = rng.standard_normal((T, 1, D))
    g = rng.uniform(-1, 0, (T, 1, D))
    h0 = rng.standard_normal((1, 1, D, D))
    r = oracle.run(q, k, v, g, np.zeros((T, 1)), [0, T], 0.5, h0=h0)
    G = np.cumsum(g[:, 0], axis=0)  # [T, D]
    for t in range(T):
        St = np.exp(G[t])[:, None] * h0[0, 0]
        np.testing.assert_allclose(r["out"][t, 0], 0.5 * St.T @ q[t, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["ht"][0, 0], np.exp(G[-1])[:, None] * h0[0, 0], rtol=1e-12)
    r0 = oracle.run(q, k, v, g, np.zeros((T, 1)), [0, T], 0.5)
    assert np.all(r0["out"] == 0.0)


def test_orthogonal_keys_reduce_to_causal_linear_attention():
    # g = 0 and orthonormal keys: r_t = v_t, so o_t = scale sum_{s<=t} beta_s (q_t.k_s) v_s.
    rng = np.random.default_rng(6)
    L, D = 12, 16
    Qm, _ = np.linalg.qr(rng.standard_normal((D, D)))
    k = Qm[:, :L].T.copy()[:, None, :]
    q = rng.standard_normal((L, 1, D)); v = rng.standard_normal((L, 1, D))
    b = rng.uniform(0, 1, (L, 1))
    r = oracle.run(q, k, v, np.zeros((L, 1, D)), b, [0, L], 0.3)
    A = np.tril(q[:, 0] @ k[:, 0].T) * b[:, 0][None, :]
    np.testing.assert_allclose(r["out"][:, 0], 0.3 * A @ v[:, 0], rtol=1e-11, atol=1e-13)


def test_orthogonal_keys_scalar_gate_decayed_attention():
    # GDN (scalar gate) keeps orthogonal keys orthogonal, so
    # o_t = scale sum_{s<=t} exp(G_t - G_s) beta_s (q_t.k_s) v_s,  G = cumsum(g).
    rng = np.random.default_rng(7)
    L, D = 10, 16
    Qm, _ = np.linalg.qr(rng.standard_normal((D, D)))
    k = Qm[:, :L].T.copy()[:, None, :]
    q = rng.standard_normal((L, 1, D)); v = rng.standard_normal((L, 1, D))
    b = rng.uniform(0, 1, (L, 1)); g = rng.uniform(-1, 0, (L, 1))
    r = oracle.run(q, k, v, g, b, [0, L], 0.3)
    G = np.cumsum(g[:, 0])
    Dm = np.tril(np.exp(G[:, None] - G[None, :]))
    A = (q[:, 0] @ k[:, 0].T) * Dm * b[:, 0][None, :]
    np.testing.assert_allclose(r["out"][:, 0], 0.3 * A @ v[:, 0], rtol=1e-11, atol=1e-13)


def test_axis_keys_per_channel_gate_decay_index():
    # KDA with keys on distinct coordinate axes: k_s = e_{p(s)}.  Decay keeps
    # each key on its axis, so r_t = v_t and channel p(s) decays by
    # exp(sum_{s<u<=t} g_{u,p(s)}):  o_t = scale sum_s beta_s q_{t,p(s)} e^{...} v_s.
    rng = np.random.default_rng(8)
    L, D = 6, 8
    perm = rng.permutation(D)[:L]
    k = np.zeros((L, 1, D)); k[np.arange(L), 0, perm] = 1.0
    q = rng.standard_normal((L, 1, D)); v = rng.standard_normal((L, 1, D))
    b = rng.uniform(0, 1, (L, 1)); g = rng.uniform(-1, 0, (L, 1, D))
    r = oracle.run(q, k, v, g, b, [0, L], 1.0)
    G = np.cumsum(g[:, 0], axis=0)
    for t in range(L):
        o = np.zeros(D)
        for s in range(t + 1):
            c = perm[s]
            o += b[s, 0] * q[t, 0, c] * np.exp(G[t, c] - G[s, c]) * v[s, 0]
        np.testing.assert_allclose(r["out"][t, 0], o, rtol=1e-11, atol=1e-13)


def test_packed_equals_per_document():
    rng = np.random.default_rng(9)
    lengths = [5, 0, 11, 1, 7]
    for per_channel, (Hqk, HV) in ((True, (2, 2)), (False, (1, 3))):
        P = _rand_problem(rng, lengths, Hqk=Hqk, HV=HV, D=8, per_channel=per_channel)
        whole = oracle.run(P["q"], P["k"], P["v"], P["g"], P["beta"], P["cu"], 0.4,
                           h0=P["h0"], dout=P["dout"], dht=P["dht"])
        cu = P["cu"]
        for n in range(len(lengths)):
            s, e = cu[n], cu[n + 1]
            one = oracle.run(P["q"][s:e], P["k"][s:e], P["v"][s:e], P["g"][s:e], P["beta"][s:e], [0, e - s], 0.4,
                             h0=P["h0"][n:n + 1], dout=P["dout"][s:e], dht=P["dht"][n:n + 1])
            for name in ("out", "dq", "dk", "dv", "dg", "dbeta"):
                assert np.array_equal(whole[name][s:e], one[name]), name
            assert np.array_equal(whole["ht"][n], one["ht"][0])
            assert np.array_equal(whole["dh0"][n], one["dh0"][0])
        # Empty document: ht = h0 and dh0 = dht.
        assert np.array_equal(whole["ht"][1], P["h0"][1])
        assert np.array_equal(whole["dh0"][1], P["dht"][1])


def test_threads_do_not_change_results():
    rng = np.random.default_rng(10)
    P = _rand_problem(rng, [30, 17, 40, 3], Hqk=2, HV=6, D=8, per_channel=False)
    a = oracle.run(P["q"], P["k"], P["v"], P["g"], P["beta"], P["cu"], 0.4, dout=P["dout"], threads=1)
    b = oracle.run(P["q"], P["k"], P["v"], P["g"], P["beta"], P["cu"], 0.4, dout=P["dout"], threads=5)
    for name in a:
        assert np.array_equal(a[name], b[name]), name


def test_kda_gdn_equivalence():
    rng = np.random.default_rng(11)
    P = _rand_problem(rng, [9, 4], Hqk=2, HV=2, D=8, per_channel=False)
    gdn = oracle.run(P["q"], P["k"], P["v"], P["g"], P["beta"], P["cu"], 0.4, h0=P["h0"], dout=P["dout"], dht=P["dht"])
    gk = np.repeat(P["g"][:, :, None], 8, axis=2)
    kda = oracle.run(P["q"], P["k"], P["v"], gk, P["beta"], P["cu"], 0.4, h0=P["h0"], dout=P["dout"], dht=P["dht"])
    for name in ("out", "ht", "dq", "dk", "dv", "dbeta", "dh0"):
        np.testing.assert_allclose(gdn[name], kda[name], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(gdn["dg"], kda["dg"].sum(-1), rtol=1e-11, atol=1e-12)


def test_grouped_gdn_equals_repeated_heads():
    rng = np.random.default_rng(12)
    P = _rand_problem(rng, [6, 5], Hqk=2, HV=6, D=4, per_channel=False)
    grouped = oracle.run(P["q"], P["k"], P["v"], P["g"], P["beta"], P["cu"], 0.4, h0=P["h0"], dout=P["dout"], dht=P["dht"])
    qr = np.repeat(P["q"], 3, axis=1)  # value head j reads Q/K head j // 3
    kr = np.repeat(P["k"], 3, axis=1)
    flat = oracle.run(qr, kr, P["v"], P["g"], P["beta"], P["cu"], 0.4, h0=P["h0"], dout=P["dout"], dht=P["dht"])
    for name in ("out", "ht", "dv", "dg", "dbeta", "dh0"):
        np.testing.assert_allclose(grouped[name], flat[name], rtol=1e-12, atol=1e-13)
    T = qr.shape[0]
    np.testing.assert_allclose(grouped["dq"], flat["dq"].reshape(T, 2, 3, 4).sum(2), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(grouped["dk"], flat["dk"].reshape(T, 2, 3, 4).sum(2), rtol=1e-12, atol=1e-13)


def test_invalid_problem_rejected():
    rng = np.random.default_rng(13)
    P = _rand_problem(rng, [3, 2], Hqk=1, HV=1, D=4, per_channel=True)
    with pytest.raises(ValueError):
        oracle.run(P["q"], P["k"], P["v"], P["g"], P["beta"], [0, 4, 5][:2] + [4], 0.4)
    with pytest.raises(ValueError):
        oracle.run(P["q"], P["k"], P["v"], P["g"], P["beta"], [0, 3, 2], 0.4)


def test_oracle_regression_fixture():
    # Frozen oracle results written by tests/golden/make_golden.py; a change to
    # the oracle's arithmetic must change this fixture in the same commit.
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_regression.json")
    with open(path) as f:
        data = json.load(f)
    for name, case in data.items():
        x = {k: np.array(v) for k, v in case["inputs"].items()}
        r = oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], case["cu_seqlens"], case["scale"],
                       h0=x["h0"], dout=x["dout"])
        for k, v in case["outputs"].items():
            np.testing.assert_allclose(r[k], np.array(v), rtol=1e-12, atol=1e-14, err_msg=f"{name}:{k}")


# In-kernel q/k L2 normalization (qk_l2norm): the recurrence runs on
# n = x (sum x^2 + eps)^(-1/2) for each (token, Q/K head) vector of q and k.
def _raw_problem(rng, lengths, Hqk, HV, D, per_channel, glow=-1.0):
    P = _rand_problem(rng, lengths, Hqk, HV, D, per_channel, glow=glow)
    # Raw, unnormalized q and k with norms far from 1.
    P["q"] = rng.standard_normal(P["q"].shape) * rng.uniform(0.2, 3.0, P["q"].shape[:2] + (1,))
    P["k"] = rng.standard_normal(P["k"].shape) * rng.uniform(0.2, 3.0, P["k"].shape[:2] + (1,))
    return P


def test_fd_gradients_with_qk_l2norm_kda():
    rng = np.random.default_rng(30)
    _check_fd(_raw_problem(rng, [5, 3], Hqk=2, HV=2, D=4, per_channel=True), scale=0.7, l2=True)


def test_fd_gradients_with_qk_l2norm_gdn_grouped():
    rng = np.random.default_rng(31)
    _check_fd(_raw_problem(rng, [4, 3], Hqk=1, HV=3, D=4, per_channel=False), scale=0.6, l2=True)


def test_qk_l2norm_is_scale_invariant_and_its_gradients_are_orthogonal():
    # Scaling a q or k vector by any positive factor leaves every output unchanged (up to
    # the epsilon), so dq . q = 0 and dk . k = 0 for every (token, head).
    rng = np.random.default_rng(32)
    P = _raw_problem(rng, [9, 6], Hqk=2, HV=4, D=8, per_channel=False)
    args = (P["v"], P["g"], P["beta"], P["cu"], 0.5)
    r = oracle.run(P["q"], P["k"], *args, h0=P["h0"], dout=P["dout"], dht=P["dht"], qk_l2norm=True)
    lam = rng.uniform(0.1, 10.0, P["q"].shape[:2] + (1,))
    mu = rng.uniform(0.1, 10.0, P["k"].shape[:2] + (1,))
    r2 = oracle.run(P["q"] * lam, P["k"] * mu, *args, h0=P["h0"], qk_l2norm=True)
    np.testing.assert_allclose(r2["out"], r["out"], rtol=1e-4, atol=1e-6)
    # (exactly zero without the epsilon; with it x . dx = r (x . dn) eps / (|x|^2 + eps))
    np.testing.assert_allclose((r["dq"] * P["q"]).sum(-1), 0.0, atol=1e-5)
    np.testing.assert_allclose((r["dk"] * P["k"]).sum(-1), 0.0, atol=1e-5)


def test_qk_l2norm_on_unit_vectors():
    # With unit q and k (and the epsilon's effect below 1e-6), the flag changes nothing in
    # the forward, and dq, dk become the flag-off gradients with their components along q,
    # k removed (the normalization's Jacobian at a unit vector is I - x x^T).
    rng = np.random.default_rng(33)
    P = _rand_problem(rng, [7, 5], Hqk=2, HV=2, D=8, per_channel=True)
    P["q"] /= np.linalg.norm(P["q"], axis=-1, keepdims=True)
    args = (P["q"], P["k"], P["v"], P["g"], P["beta"], P["cu"], 0.8)
    off = oracle.run(*args, h0=P["h0"], dout=P["dout"], dht=P["dht"])
    on = oracle.run(*args, h0=P["h0"], dout=P["dout"], dht=P["dht"], qk_l2norm=True)
    for name in ("out", "ht", "dv", "dg", "dbeta", "dh0"):
        np.testing.assert_allclose(on[name], off[name], rtol=2e-6, atol=2e-6)
    for x, gname in (("q", "dq"), ("k", "dk")):
        u = P[x]
        proj = off[gname] - u * (u * off[gname]).sum(-1, keepdims=True)
        np.testing.assert_allclose(on[gname], proj, rtol=2e-6, atol=2e-6)
