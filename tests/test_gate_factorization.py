"""The per-channel gate factorization of the KDA kernels, emulated in FP32 on
the CPU: within a 64-token chunk the decays exp(gc_i - gc_j) of the gated Gram
matrix are split per 16-row block around one reference, the block's 8th row,
so that every factor stays finite in FP32 for gates down to the library's
bound of -10 per token, where splitting around the chunk start overflows.
(The GPU parity tests run the kernels themselves on gates down to -10.)"""
import numpy as np
import pytest

CH, BLOCK = 64, 16


def _exact(K, gc):
    """At[i][j] = sum_c K_ic K_jc exp(gc_ic - gc_jc), j < i, in FP64."""
    K, gc = K.astype(np.float64), gc.astype(np.float64)
    d = gc[:, None, :] - gc[None, :, :]  # |d| <= 640 here: exp(d) is finite in FP64
    return np.tril(np.einsum("ic,jc,ijc->ij", K, K, np.exp(d)), -1)


def _blocked_fp32(K, gc):
    """Row block I: A = K_I exp(gc_I - r), B = K_j exp(r - gc_j) for j < 16 I + 16,
    r = gc at row 16 I + 7; every operation in FP32.  Each factor must be
    finite (checked); their products above the diagonal of a diagonal block,
    exp(gc_i - gc_j) with i < j, may overflow and are dropped by select, as
    the kernels mask them."""
    K, gc = K.astype(np.float32), gc.astype(np.float32)
    At = np.zeros((CH, CH), np.float32)
    for I in range(CH // BLOCK):
        i0 = BLOCK * I
        r = gc[i0 + 7]
        with np.errstate(over="raise", invalid="raise"):
            A = K[i0:i0 + BLOCK] * np.exp(gc[i0:i0 + BLOCK] - r)
            B = K[:i0 + BLOCK] * np.exp(r - gc[:i0 + BLOCK])
        with np.errstate(over="ignore", invalid="ignore"):
            At[i0:i0 + BLOCK, :i0 + BLOCK] = A @ B.T
    keep = np.tril(np.ones((CH, CH), bool), -1)
    return np.where(keep, At, np.float32(0.0))


def _chunk(seed, glow, D=32):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((CH, D))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    g = rng.uniform(glow, 0.0, (CH, D))
    g[:, 0] = glow  # one channel at the bound on every token
    gc = np.cumsum(g.astype(np.float32), axis=0, dtype=np.float32)
    return K.astype(np.float32), gc


@pytest.mark.parametrize("glow", [-0.1, -1.0, -5.0, -10.0])
def test_block_factorization_is_finite_and_accurate_in_fp32(glow):
    K, gc = _chunk(3, glow)
    got = _blocked_fp32(K, gc)
    ref = _exact(K, gc)
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 1e-5 * max(np.abs(ref).max(), 1.0)


def test_splitting_around_the_chunk_start_overflows():
    # exp(gc_i) exp(-gc_j) with gc from the chunk start: -gc reaches 640 at
    # g = -10, far beyond FP32's largest finite value (about exp(88.7)).
    K, gc = _chunk(3, -10.0)
    with np.errstate(over="ignore", invalid="ignore"):
        naive = np.tril((K * np.exp(gc)) @ (K * np.exp(-gc)).T, -1)
    assert not np.isfinite(naive).all()
