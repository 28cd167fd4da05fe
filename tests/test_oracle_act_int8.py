"""Pins of the oracle's INT4 x int8-activation GEMV (CPU): activations already on the int8 grid
reduce it to the plain dequantized GEMV (a library matmul), hand-checked ties and zero groups,
and the rounding bound against the exact product."""
import numpy as np

from oracle import act_int8 as oa
from oracle import quantize as oq


def _weights(seed, N, K):
    rng = np.random.default_rng(seed)
    codes = rng.integers(-8, 8, (N, K)).astype(np.int8)
    sbits = oq.bf16_rne_bits(rng.uniform(0.002, 0.006, (N, K // 128)).astype(np.float32))
    return codes, sbits


def _dense(codes, sbits):
    sw = np.repeat(oq.bf16_bits_to_f32(sbits).astype(np.float64), 128, axis=1)
    return codes.astype(np.float64) * sw


def test_activations_on_the_grid_give_the_dequantized_gemv():
    rng = np.random.default_rng(1)
    N, K = 48, 512
    codes, sbits = _weights(2, N, K)
    q = rng.integers(-127, 128, K)
    q[::128] = 127                                       # every group reaches 127: sx = 2^-7 exactly
    x = (q * 2.0 ** -7).astype(np.float32)
    qq, sx = oa.quantize_activations_g128(x)
    assert np.all(sx == np.float32(2.0 ** -7)) and np.array_equal(qq, q)
    y, _ = oa.gemv_int4_a8(codes, sbits, x)
    want = _dense(codes, sbits) @ x.astype(np.float64)
    assert np.allclose(y, want, rtol=1e-12, atol=0)


def test_ties_and_zero_groups():
    x = np.zeros(256, np.float32)
    x[:4] = [127.0, 2.5, -3.5, 0.5]                      # sx = 1
    q, sx = oa.quantize_activations_g128(x)
    assert sx[0] == 1.0 and sx[1] == 0.0
    assert list(q[:4]) == [127, 2, -4, 0] and not q[128:].any()
    codes = np.zeros((1, 256), np.int8)
    codes[0, :4] = [1, 1, 1, 1]
    codes[0, 200] = 7                                    # meets the zero group: contributes 0
    sbits = oq.bf16_rne_bits(np.array([[0.5, 0.25]], np.float32))
    y, _ = oa.gemv_int4_a8(codes, sbits, x)
    assert y[0] == 0.5 * 1.0 * (127 + 2 - 4 + 0)


def test_rounding_bound_against_the_exact_product():
    rng = np.random.default_rng(3)
    N, K = 64, 1024
    codes, sbits = _weights(4, N, K)
    x = rng.normal(0, 1, K).astype(np.float32)
    y, _ = oa.gemv_int4_a8(codes, sbits, x)
    exact = _dense(codes, sbits) @ x.astype(np.float64)
    _, sx = oa.quantize_activations_g128(x)
    sw = oq.bf16_bits_to_f32(sbits).astype(np.float64)
    bound = (sw * sx[None, :] * 0.5 * np.abs(codes.astype(np.float64)).reshape(N, -1, 128).sum(axis=2)).sum(axis=1)
    err = np.abs(y - exact)
    assert np.all(err <= bound * (1 + 1e-6))
    assert err.max() > 0                                 # the activations were rounded
