"""CPU oracle of the offline weight quantizers.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's CPU baseline
leg may import this module.  The library never does; the two share no code.

  * INT4, group 128 ["How To Construct Your Personal LLM Runtime From Scratch", §3: symmetric
    group-wise INT4, group size 128, one scale per group per output row, scale = absmax / 7,
    zero point 0]: scale_fp32 = absmax / 7, stored as bfloat16 (round to nearest, ties to even).
  * INT8, per row ["FlashQwen", Stage 8: symmetric INT8 with one scale per output row, computed
    at load]: scale = absmax / 127 (fp32).
Reading (the pages do not say): each code is the fp32 quotient weight / scale, with the scale as
it is stored, rounded half to even and clamped to the format's range ([-8, 7], [-127, 127]);
an all-zero group or row has scale 0 and codes 0.  The quotient decides an integer, so it is
taken in fp32 here as in the library.
"""
import numpy as np


def bf16_rne_bits(x):
    """fp32 -> bfloat16 bit pattern, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def quantize_int4_g128(w):
    """w fp32 [N][K] (K % 128 == 0) -> codes int8 [N][K], scale bits uint16 [N][K/128]."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    g = w.reshape(N, K // 128, 128)
    amax = np.abs(g).max(axis=2)
    sbits = bf16_rne_bits(amax / np.float32(7.0))
    s = bf16_bits_to_f32(sbits)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(g / s)
    q = np.where(s > 0, np.clip(q, -8, 7), 0).astype(np.int8)
    return q.reshape(N, K), sbits


def quantize_int8_row(w):
    """w fp32 [N][K] -> codes int8 [N][K], scales fp32 [N]."""
    w = np.asarray(w, dtype=np.float32)
    s = np.abs(w).max(axis=1) / np.float32(127.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(w / s[:, None])
    q = np.where(s[:, None] > 0, np.clip(q, -127, 127), 0).astype(np.int8)
    return q, s.astype(np.float32)
