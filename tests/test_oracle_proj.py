"""Pins of the fp64 QKV-projection oracle (CPU, no GPU).

Each check is fixed by the definition (a linear layer with one concatenated
q/k/v weight, q block scaled by HD^-0.5), not by retyping the oracle's
formula: explicit sums on tiny inputs, an identity weight, a zero input, the
block order of q, k and v, and linearity.
"""
import numpy as np
import pytest

import na3d_inputs
import oracle


def bits(a):
    return na3d_inputs.f64_to_bf16_bits(np.asarray(a, dtype=np.float64))


def test_explicit_sums_on_tiny_inputs():
    rng = np.random.default_rng(1)
    M, C, NH, HD = 3, 5, 1, 16
    N = 3 * NH * HD
    x, w, b = bits(rng.normal(size=(M, C))), bits(rng.normal(size=(N, C))), bits(rng.normal(size=N))
    xf = na3d_inputs.bf16_bits_to_f64(x)
    wf = na3d_inputs.bf16_bits_to_f64(w)
    bf = na3d_inputs.bf16_bits_to_f64(b)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for c in range(C):
                s += xf[m, c] * wf[n, c]
            s += bf[n]
            want[m, n] = s / 4.0 if n < NH * HD else s   # HD = 16: scale 1/4
    np.testing.assert_allclose(oracle.qkv_projection(x, w, b, NH, HD), want, rtol=1e-14, atol=1e-14)


def test_identity_weight_returns_x_with_the_q_block_scaled():
    NH, HD = 2, 16
    N = 3 * NH * HD
    rng = np.random.default_rng(2)
    x = bits(rng.normal(size=(7, N)))
    got = oracle.qkv_projection(x, bits(np.eye(N)), None, NH, HD)
    xf = na3d_inputs.bf16_bits_to_f64(x)
    np.testing.assert_array_equal(got[:, :NH * HD], xf[:, :NH * HD] * 0.25)
    np.testing.assert_array_equal(got[:, NH * HD:], xf[:, NH * HD:])


def test_zero_input_returns_the_bias_with_the_q_block_scaled():
    NH, HD, C = 3, 64, 24
    N = 3 * NH * HD
    b = bits(np.linspace(-3, 3, N))
    got = oracle.qkv_projection(bits(np.zeros((4, C))), bits(np.ones((N, C))), b, NH, HD)
    bf = na3d_inputs.bf16_bits_to_f64(b)
    np.testing.assert_array_equal(got[0, :NH * HD], bf[:NH * HD] * 0.125)
    np.testing.assert_array_equal(got[2, NH * HD:], bf[NH * HD:])


def test_block_order_q_then_k_then_v():
    """Weight rows r of block j pick input channel j: the q, k and v blocks of
    the output hold channels 0, 1 and 2 (q scaled)."""
    NH, HD, C = 1, 16, 3
    N = 3 * NH * HD
    w = np.zeros((N, C))
    for j in range(3):
        w[j * NH * HD:(j + 1) * NH * HD, j] = 1.0
    x = bits([[5.0, 7.0, 11.0]])
    got = oracle.qkv_projection(x, bits(w), None, NH, HD)[0]
    assert np.all(got[:16] == 1.25) and np.all(got[16:32] == 7.0) and np.all(got[32:] == 11.0)


@pytest.mark.parametrize("HD", [16, 32, 64, 128])
def test_linear_in_x(HD):
    """Doubling x is exact in bf16, so f(2x) = 2 f(x) - f(0) (the bias once)."""
    rng = np.random.default_rng(HD)
    NH, C = 2, 40
    N = 3 * NH * HD
    w, b = bits(rng.normal(size=(N, C))), bits(rng.normal(size=N))
    x = rng.normal(size=(5, C))
    f = lambda xx: oracle.qkv_projection(bits(xx), w, b, NH, HD)   # noqa: E731
    xr = na3d_inputs.bf16_bits_to_f64(bits(x))                      # x as bf16 values
    np.testing.assert_allclose(f(2 * xr), 2 * f(xr) - f(np.zeros_like(xr)), rtol=1e-12, atol=1e-12)
