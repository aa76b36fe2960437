"""The chunked identities the kernels implement, checked in FP64 against the
oracle's token-by-token recurrence (CPU).

Per chunk of C tokens (rows i, gc = chunk-local cumsum of the log-decay,
Gamma = exp(gc), gamma = Gamma at the chunk's last row, Kd = K exp(gc_last - gc)):

  At  = strict_tril((K Gamma) (K / Gamma)^T),   T = (I + diag(beta) At)^-1
  w   = T diag(beta) (K Gamma),  u = T diag(beta) V,   Delta = u - w S0
  Aqk = tril((Q Gamma) (K / Gamma)^T)
  O   = scale ((Q Gamma) S0 + Aqk Delta),   S_end = diag(gamma) S0 + Kd^T Delta

and the backward from dO and dS (the adjoint of S_end):

  dDelta = scale Aqk^T dO + Kd dS,   dS0 = diag(gamma) dS + scale (Q Gamma)^T dO - w^T dDelta
  dAqk = scale tril(dO Delta^T),  X = T^T (-dDelta S0^T),  Y = T^T dDelta
  dA = -strict_tril(X w^T + Y u^T)
  dQ = scale (dO S0^T) Gamma + Gamma (dAqk (K / Gamma))
  dKp = beta X Gamma + beta Gamma (dA (K / Gamma))              (the K Gamma occurrences)
  dKn = (dAqk^T (Q Gamma) + (diag(beta) dA)^T (K Gamma)) / Gamma (the K / Gamma occurrences)
  dV = beta Y,   dbeta = rowsum(X K Gamma) + rowsum(Y V) + rowsum(dA At)
  dKd = Delta dS^T,   dK = dKp + dKn + dKd gamma / Gamma
  dgc = Q dQ + K dKp - K dKn - Kd dKd, and at the last row
        + gamma rowsum(dS S0) + colsum(Kd dKd);   dg = reverse cumsum of dgc.

Nothing here is shared with the oracle or the CUDA path: this is the chunked
algorithm written out once more, so that a mistake in the identities the
kernels follow (a dropped term, a wrong transpose or mask) fails against the
oracle without a GPU.  FP64 throughout, so the gates are split as
exp(gc_i) exp(-gc_j) directly (the kernels factor them per 16-row block).
"""
import numpy as np
import pytest

import oracle


def _chunk_fwd(Q, K, V, G, beta, S0, scale):
    L = Q.shape[0]
    gc = np.cumsum(G, axis=0)
    Gam = np.exp(gc)
    Kp, Kn, Qp = K * Gam, K / Gam, Q * Gam
    At = np.tril(Kp @ Kn.T, -1)
    Tm = np.linalg.inv(np.eye(L) + beta[:, None] * At)
    w = Tm @ (beta[:, None] * Kp)
    u = Tm @ (beta[:, None] * V)
    Delta = u - w @ S0
    Aqk = np.tril(Qp @ Kn.T)
    O = scale * (Qp @ S0 + Aqk @ Delta)
    gamma = Gam[-1]
    Kd = K * gamma / Gam
    S_end = gamma[:, None] * S0 + Kd.T @ Delta
    saved = dict(Q=Q, K=K, V=V, beta=beta, S0=S0, Gam=Gam, Kp=Kp, Kn=Kn, Qp=Qp, At=At, Tm=Tm, w=w, u=u,
                 Delta=Delta, Aqk=Aqk, gamma=gamma, Kd=Kd)
    return O, S_end, saved


def _chunk_bwd(s, dO, dS, scale):
    Q, K, V, beta, S0 = s["Q"], s["K"], s["V"], s["beta"], s["S0"]
    Gam, Kp, Kn, Qp, At, Tm = s["Gam"], s["Kp"], s["Kn"], s["Qp"], s["At"], s["Tm"]
    w, u, Delta, Aqk, gamma, Kd = s["w"], s["u"], s["Delta"], s["Aqk"], s["gamma"], s["Kd"]
    dDelta = scale * Aqk.T @ dO + Kd @ dS
    dS0 = gamma[:, None] * dS + scale * Qp.T @ dO - w.T @ dDelta
    dAqk = scale * np.tril(dO @ Delta.T)
    X = Tm.T @ (-dDelta @ S0.T)
    Y = Tm.T @ dDelta
    dA = -np.tril(X @ w.T + Y @ u.T, -1)
    dQ = scale * (dO @ S0.T) * Gam + Gam * (dAqk @ Kn)
    dKp = beta[:, None] * X * Gam + beta[:, None] * Gam * (dA @ Kn)
    dKn = (dAqk.T @ Qp + (beta[:, None] * dA).T @ Kp) / Gam
    dV = beta[:, None] * Y
    dbeta = (X * Kp).sum(1) + (Y * V).sum(1) + (dA * At).sum(1)
    dKd = Delta @ dS.T
    dK = dKp + dKn + dKd * gamma / Gam
    dgc = Q * dQ + K * dKp - K * dKn - Kd * dKd
    dgc[-1] += gamma * (dS * S0).sum(1) + (Kd * dKd).sum(0)
    dG = np.cumsum(dgc[::-1], axis=0)[::-1]
    return dQ, dK, dV, dG, dbeta, dS0


def chunked(q, k, v, g, beta, cu, scale, h0, dout, dht, C):
    """Forward and backward of a packed problem by the chunked identities."""
    T, Hqk, D = q.shape
    HV = v.shape[1]
    per_channel = g.ndim == 3
    gf = g if per_channel else np.repeat(g[:, :, None], D, axis=2)
    out = np.zeros((T, HV, D))
    N = len(cu) - 1
    ht = np.zeros((N, HV, D, D))
    dq, dk = np.zeros((T, Hqk, D)), np.zeros((T, Hqk, D))
    dv, dgf, dbeta = np.zeros((T, HV, D)), np.zeros((T, HV, D)), np.zeros((T, HV))
    dh0 = np.zeros((N, HV, D, D))
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(HV):
            hq = h // (HV // Hqk)
            S = h0[n, h].copy()
            tape = []
            for c0 in range(t0, t1, C):
                c1 = min(c0 + C, t1)
                O, S, sv = _chunk_fwd(q[c0:c1, hq], k[c0:c1, hq], v[c0:c1, h], gf[c0:c1, h], beta[c0:c1, h], S, scale)
                out[c0:c1, h] = O
                tape.append((c0, c1, sv))
            ht[n, h] = S
            dS = dht[n, h].copy()
            for c0, c1, sv in reversed(tape):
                dQ, dK, dV, dG, dB, dS = _chunk_bwd(sv, dout[c0:c1, h], dS, scale)
                dq[c0:c1, hq] += dQ
                dk[c0:c1, hq] += dK
                dv[c0:c1, h] = dV
                dgf[c0:c1, h] = dG
                dbeta[c0:c1, h] = dB
            dh0[n, h] = dS
    dg = dgf if per_channel else dgf.sum(axis=2)
    return dict(out=out, ht=ht, dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dh0=dh0)


def _problem(seed, lengths, Hqk, HV, D, per_channel, glow):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    q = rng.standard_normal((T, Hqk, D))
    k = rng.standard_normal((T, Hqk, D))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, HV, D))
    g = rng.uniform(glow, 0.0, (T, HV, D) if per_channel else (T, HV))
    beta = rng.uniform(0.0, 1.0, (T, HV))
    N = len(lengths)
    h0 = rng.standard_normal((N, HV, D, D))
    dout = rng.standard_normal((T, HV, D))
    dht = rng.standard_normal((N, HV, D, D))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, g, beta, cu, h0, dout, dht


# Ragged documents: several full chunks and a tail, exactly one chunk, one
# token, an empty document, a chunk plus a few tokens.
LENGTHS = [150, 64, 1, 0, 70]


@pytest.mark.parametrize("C", [64, 16])
@pytest.mark.parametrize(
    "Hqk,HV,per_channel,glow",
    [(2, 2, True, -1.0),   # KDA: per-channel gate
     (2, 2, False, -2.0),  # GDN: scalar gate
     (1, 3, False, -0.5)],  # grouped GDN: three value heads per Q/K head
)
def test_chunked_identities_match_the_recurrence(C, Hqk, HV, per_channel, glow):
    q, k, v, g, beta, cu, h0, dout, dht = _problem(7, LENGTHS, Hqk, HV, 8, per_channel, glow)
    scale = 0.35
    ref = oracle.run(q, k, v, g, beta, cu, scale, h0=h0, dout=dout, dht=dht)
    got = chunked(q, k, v, g, beta, cu, scale, h0, dout, dht, C)
    for name in ("out", "ht", "dq", "dk", "dv", "dg", "dbeta", "dh0"):
        a, b = got[name], ref[name]
        err = np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)
        assert err < 1e-10, f"{name}: chunked identities differ from the recurrence by {err:.2e}"


def _walk(q, k, v, g, beta, S, scale, C):
    """One (document, head) chain of chunks from S: (end state, per-chunk saved values)."""
    tape = []
    for c0 in range(0, q.shape[0], C):
        c1 = min(c0 + C, q.shape[0])
        _, S, sv = _chunk_fwd(q[c0:c1], k[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1], S, scale)
        tape.append((c0, c1, sv))
    return S, tape


def _walk_back(tape, dout, dS, scale):
    for c0, c1, sv in reversed(tape):
        dS = _chunk_bwd(sv, dout[c0:c1], dS, scale)[5]
    return dS


@pytest.mark.parametrize("per_channel", [True, False])
def test_segment_maps_are_affine(per_channel):
    # A run of chunks maps its start state affinely, S_end = M S_start + B, with
    # M the end state walked from the identity with v = 0 (so u = 0) and B the
    # end state walked from zero; its adjoint maps back as
    # dS_start = M^T dS_end + dB, with dB walked back from a zero end adjoint.
    # The segment-parallel walks (summary walks, then a merge) rest on these.
    rng = np.random.default_rng(11)
    L, D, scale = 200, 8, 0.4
    q = rng.standard_normal((L, D))
    k = rng.standard_normal((L, D))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((L, D))
    g = rng.uniform(-0.2, 0.0, (L, D)) if per_channel else np.repeat(rng.uniform(-0.2, 0.0, (L, 1)), D, 1)
    beta = rng.uniform(0.0, 1.0, L)
    dout = rng.standard_normal((L, D))
    S_start, dS_end = rng.standard_normal((D, D)), rng.standard_normal((D, D))
    M, _ = _walk(q, k, np.zeros_like(v), g, beta, np.eye(D), scale, 64)
    B, tape0 = _walk(q, k, v, g, beta, np.zeros((D, D)), scale, 64)
    S_end, tape = _walk(q, k, v, g, beta, S_start, scale, 64)
    assert np.abs(S_end - (M @ S_start + B)).max() < 1e-12 * max(1.0, np.abs(S_end).max())
    dB = _walk_back(tape0, dout, np.zeros((D, D)), scale)
    dS_start = _walk_back(tape, dout, dS_end, scale)
    assert np.abs(dS_start - (M.T @ dS_end + dB)).max() < 1e-12 * max(1.0, np.abs(dS_start).max())
