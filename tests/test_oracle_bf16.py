"""Pins of the oracle's dense BF16 steps (router GEMM, latent projections,
shared-expert MLP).

- orc_gemm_bf16 against numpy's fp64 matmul of the decoded bf16 operands (an
  independent library routine) on ragged shapes, and against a brute-force
  Python double loop on a tiny one; transposition and operand order pinned
  by a non-square case with distinct rows.
- Closed forms: an identity B gives A back exactly; a one-hot A row picks one
  column of B^T; bf16 decoding exact for special values.
- orc_gemm_bf16_swiglu: silu(g) * u against scipy's expit on the same
  products, gate rows first (swapping the halves changes the result).
"""
import numpy as np
import torch
from scipy.special import expit

from tests import mx_numpy as mx


def _bf16(x):
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_gemm_matches_numpy_matmul(orc):
    g = np.random.default_rng(0)
    for M, N, K in ((7, 13, 64), (33, 5, 192), (1, 96, 128)):
        a = _bf16(g.standard_normal((M, K)))
        b = _bf16(g.standard_normal((N, K)) * 0.1)
        ref = mx.bf16_bits_to_f64(a) @ mx.bf16_bits_to_f64(b).T
        got = orc.gemm_bf16(a, b)
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_gemm_brute_force_tiny(orc):
    g = np.random.default_rng(1)
    a = _bf16(g.standard_normal((3, 4)))
    b = _bf16(g.standard_normal((2, 4)))
    A, B = mx.bf16_bits_to_f64(a), mx.bf16_bits_to_f64(b)
    got = orc.gemm_bf16(a, b)
    for m in range(3):
        for n in range(2):
            s = 0.0
            for t in range(4):
                s += A[m, t] * B[n, t]
            assert abs(got[m, n] - s) <= 1e-15 * (abs(s) + 1)
    assert got.shape == (3, 2)


def test_gemm_closed_forms(orc):
    g = np.random.default_rng(2)
    K = 64
    a = _bf16(g.standard_normal((5, K)))
    eye = _bf16(np.eye(K))
    np.testing.assert_array_equal(orc.gemm_bf16(a, eye), mx.bf16_bits_to_f64(a))
    b = _bf16(g.standard_normal((9, K)))
    onehot = _bf16(np.eye(K)[[3]])
    np.testing.assert_array_equal(orc.gemm_bf16(onehot, b)[0], mx.bf16_bits_to_f64(b)[:, 3])
    special = np.array([[0.0, -0.0, 1e-40, 3.0e38, -2.5, 0.5] + [0.0] * (K - 6)], np.float32)
    one = _bf16(np.eye(K)[:6])
    got = orc.gemm_bf16(_bf16(special), one)[0]
    np.testing.assert_array_equal(got, mx.bf16_bits_to_f64(_bf16(special))[0, :6])


def test_swiglu_gate_rows_first(orc):
    g = np.random.default_rng(3)
    M, Nh, K = 6, 16, 128
    a = _bf16(g.standard_normal((M, K)))
    b = _bf16(g.standard_normal((2 * Nh, K)) * 0.2)
    A, B = mx.bf16_bits_to_f64(a), mx.bf16_bits_to_f64(b)
    G, U = A @ B[:Nh].T, A @ B[Nh:].T
    got = orc.gemm_bf16_swiglu(a, b)
    np.testing.assert_allclose(got, G * expit(G) * U, rtol=1e-12, atol=1e-14)
    swapped = orc.gemm_bf16_swiglu(a, np.concatenate([b[Nh:], b[:Nh]]))
    assert not np.allclose(swapped, got)
