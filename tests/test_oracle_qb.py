"""Pins of the oracle's integer-coded product (oracle.gemm_qb): B given as
int8 codes q_kj with one fp32 scale s_j per column, b_kj = s_j * q_kj
(Tolk.Stage, "Decoded panels on the host", read as per-column scaled int8
codes).  Each pin is fixed by something other than the oracle: numpy's fp64
matmul, closed forms, and the full range of the two's-complement code."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f16_bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


@pytest.mark.parametrize("seed", range(6))
def test_matches_numpy_fp64_matmul(seed):
    """Random shapes with row padding in A and Q, codes over the whole int8
    range, scales of both signs and many magnitudes: the fp64 value equals
    numpy's (A @ (Q * s)) and the fp16 / fp32 outputs are its RNE rounding
    as numpy's casts give it."""
    rng = np.random.default_rng(100 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 40, 3))
    lda, ldq = K + int(rng.integers(0, 5)), N + int(rng.integers(0, 5))
    a = rng.standard_normal((M, lda)).astype(np.float16)
    q = rng.integers(-128, 128, (K, ldq), dtype=np.int16).astype(np.int8)
    s = (rng.standard_normal(ldq) * 2.0 ** rng.integers(-12, 4, ldq)).astype(np.float32)
    ref = a[:, :K].astype(np.float64) @ (q[:, :N].astype(np.float64) * s[:N].astype(np.float64))
    S_ref = np.abs(a[:, :K].astype(np.float64)) @ np.abs(q[:, :N].astype(np.float64) * s[:N].astype(np.float64))
    for out in ("f32", "f16"):
        C, exact, S = oracle.gemm_qb(a.view(np.uint16), q, s, "f16", out, K=K, N=N)
        np.testing.assert_allclose(exact, ref, rtol=1e-13, atol=1e-300)
        np.testing.assert_allclose(S, S_ref, rtol=1e-13, atol=1e-300)
        want = ref.astype(np.float32).view(np.uint32) if out == "f32" else ref.astype(np.float16).view(np.uint16)
        assert np.array_equal(C, want)


def test_diagonal_closed_form():
    """Q = c I (K = N) and s_j = 2^-j: C_ij = c * 2^-j * a_ij exactly."""
    n, c = 24, -7
    rng = np.random.default_rng(7)
    a = rng.standard_normal((5, n)).astype(np.float16)
    q = (np.eye(n) * c).astype(np.int8)
    s = (2.0 ** -np.arange(n)).astype(np.float32)
    _, exact, _ = oracle.gemm_qb(a.view(np.uint16), q, s, "f16", "f32")
    assert np.array_equal(exact, a.astype(np.float64) * c * s.astype(np.float64))


def test_every_code_decodes_twos_complement():
    """One-hot rows of A pick single codes: every value -128..127 comes back
    as itself times its column's scale (an unsigned or offset decode fails)."""
    codes = np.arange(-128, 128, dtype=np.int16).astype(np.int8).reshape(16, 16)
    a = np.eye(16, dtype=np.float16)
    s = np.full(16, 0.25, dtype=np.float32)
    _, exact, _ = oracle.gemm_qb(a.view(np.uint16), codes, s, "f16", "f32")
    assert np.array_equal(exact, codes.astype(np.float64) * 0.25)


def test_bias_relu_and_zero_a():
    """A = 0: C = relu(bias) for bias_relu (the epilogue's closed form), and
    bf16 operands take the same path."""
    N, K = 9, 13
    a = np.zeros((3, K), dtype=np.uint16)
    q = np.full((K, N), 5, dtype=np.int8)
    s = np.ones(N, dtype=np.float32)
    bias = np.linspace(-2.0, 2.0, N).astype(np.float32)
    for in_dt in ("f16", "bf16"):
        _, exact, _ = oracle.gemm_qb(a, q, s, in_dt, "f32", "bias_relu", bias=bias)
        assert np.array_equal(exact, np.broadcast_to(np.maximum(bias.astype(np.float64), 0.0), (3, N)))


def test_scale_is_per_column_and_exact():
    """Doubling one column's scale doubles exactly that column."""
    rng = np.random.default_rng(9)
    a = rng.standard_normal((6, 20)).astype(np.float16).view(np.uint16)
    q = rng.integers(-100, 100, (20, 8), dtype=np.int16).astype(np.int8)
    s = rng.uniform(0.01, 1.0, 8).astype(np.float32)
    _, e1, _ = oracle.gemm_qb(a, q, s, "f16", "f32")
    s2 = s.copy()
    s2[3] *= 2
    _, e2, _ = oracle.gemm_qb(a, q, s2, "f16", "f32")
    assert np.array_equal(e2[:, 3], 2 * e1[:, 3])
    assert np.array_equal(np.delete(e2, 3, axis=1), np.delete(e1, 3, axis=1))
