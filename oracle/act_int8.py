"""CPU oracle of the INT4 GEMV on int8 activations (the opt-in decode variant).

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's CPU baseline
leg may import this module.  The library never does; the two share no code.

["How To Construct Your Personal LLM Runtime From Scratch", §7, Path A]: the activations are
quantized to INT8 with a per-group activation scale before the GEMV, the products are INT8 dot
products (__dp4a), and the group scales de-quantize inside the accumulator.
Reading (the page gives no formula): the groups are the weights' groups of 128 along K;
sx[g] = max |x| over the group / 127 in fp32; q = x / sx rounded half to even in fp32 (the
quotient decides an integer, so it is taken in the precision the GPU uses), clamped to
[-127, 127]; a zero group has sx = 0 and codes 0.  Then
    y[n] = sum_g s_w[n][g] * sx[g] * sum_{k in g} c[n][k] * q[k],
with the inner sums exact integers and the rest in float64 here.
"""
import numpy as np


def quantize_activations_g128(x):
    """x fp32 [K] (K % 128 == 0) -> codes int32 [K], scales fp32 [K/128]."""
    x = np.asarray(x, dtype=np.float32)
    g = x.reshape(-1, 128)
    sx = np.abs(g).max(axis=1) / np.float32(127.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(g / sx[:, None])
    q = np.where(sx[:, None] > 0, np.clip(q, -127, 127), 0).astype(np.int64)
    return q.reshape(-1), sx.astype(np.float32)


def gemv_int4_a8(codes, scale_bits, x):
    """codes int8 [N][K] in [-8, 7], scale_bits bf16 bit patterns [N][K/128], x fp32 [K]
    -> (y float64 [N], sum_g |s_w sx| sum_k |c q| per row, a scale for error bounds)."""
    codes = np.asarray(codes, dtype=np.int64)
    N, K = codes.shape
    q, sx = quantize_activations_g128(x)
    prod = codes.reshape(N, K // 128, 128) * q.reshape(1, K // 128, 128)
    dots = prod.sum(axis=2)                                        # exact integers
    sw = (np.asarray(scale_bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    ss = sw * sx.astype(np.float64)[None, :]
    return (ss * dots).sum(axis=1), (np.abs(ss) * np.abs(prod).sum(axis=2)).sum(axis=1)
