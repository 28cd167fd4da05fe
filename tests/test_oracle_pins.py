"""Pins of the CPU oracle against what the pages and the mathematics fix (CPU only).

Each test is chosen so that a plausible slip in the oracle (a wrong lane map, a dropped
term, a transposed operand, a wrong head-to-group map, interleaved instead of half-split
RoPE pairs) fails it.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth
from synth import model as sm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BF16_ONE = 0x3F80


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.strip() for l in f if l.strip() and not l.startswith("#")]


# ---------------------------------------------------------------- generator


def test_splitmix64_reference_vector():
    want = [int(x) for x in _golden_lines("splitmix64_seed1234567.txt")]
    got = synth.raw_state(1234567, 5).tolist()
    assert got == want


def test_generator_is_counter_based_and_ranged():
    a = synth.randint_i8(7, 3, 100_000, -8, 7)
    assert a.min() == -8 and a.max() == 7
    # every value equally likely (chi-square, 15 dof, loose bound)
    counts = np.bincount(a.astype(np.int64) + 8, minlength=16)
    exp = a.size / 16
    assert ((counts - exp) ** 2 / exp).sum() < 60
    b = synth.randint_i8(7, 3, 1000, -8, 7)
    assert np.array_equal(a[:1000], b)
    z = synth.normal_f32(1, 2, 200_000, 0.0, 1.0)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    p = synth.permutation(5, 6, 1000)
    assert np.array_equal(np.sort(p), np.arange(1000))


# ---------------------------------------------------------------- packing


def test_valueshuffle_golden_words():
    for line in _golden_lines("valueshuffle_words.txt"):
        lhs, rhs = line.split(":")
        codes = np.array([int(v) for v in lhs.split()], dtype=np.int8).reshape(1, 8)
        want = int(rhs.strip(), 16)
        words = oracle.pack_int4(codes)
        assert int(words[0, 0]) == want, line
        assert np.array_equal(oracle.unpack_int4(words), codes), line


def test_pack_unpack_round_trip_exact():
    codes = synth.randint_i8(11, 1, 64 * 1024, -8, 7).reshape(64, 1024)
    words = oracle.pack_int4(codes)
    assert words.shape == (64, 128) and words.dtype == np.uint32
    assert np.array_equal(oracle.unpack_int4(words), codes)


def test_pack_single_lane_positions():
    # a single code at lane i of word w lands at bit shift table[i] of word w only
    table = [0, 16, 4, 20, 8, 24, 12, 28]
    for w in range(3):
        for i in range(8):
            codes = np.zeros((1, 24), np.int8)
            codes[0, 8 * w + i] = 5
            words = oracle.pack_int4(codes)
            want = np.zeros(3, np.uint32)
            want[w] = 5 << table[i]
            assert np.array_equal(words[0], want)


# ---------------------------------------------------------------- bf16 storage


def test_bf16_round_ties_to_even_and_matches_torch():
    torch = pytest.importorskip("torch")
    assert oracle.bf16_round(np.float32(1.0)) == 0x3F80
    assert oracle.bf16_round(np.float32(1.0 + 2 ** -8)) == 0x3F80          # tie -> even
    assert oracle.bf16_round(np.float32(1.0 + 3 * 2 ** -8)) == 0x3F82      # tie -> even
    assert oracle.bf16_round(np.float32(1.0 + 2 ** -8 + 2 ** -20)) == 0x3F81
    assert oracle.bf16_round(np.float32(-2.0)) == 0xC000
    x = synth.normal_f32(3, 4, 4096, 0.0, 3.0)
    ours = oracle.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- RMSNorm


@pytest.mark.parametrize("prec", ["f32", "f64"])
def test_rmsnorm_closed_form(prec):
    o = oracle.Oracle(prec)
    gam = np.full(64, BF16_ONE, np.uint16)
    for c in (0.5, -3.0, 1e-3):
        y = o.rmsnorm(np.full(64, c), gam, 1e-6)
        np.testing.assert_allclose(y, c / math.sqrt(c * c + 1e-6), rtol=2e-6)
    # with eps = 0 the output has unit mean square and is scale invariant
    x = synth.normal_f32(1, 1, 256, 0.0, 2.0).astype(np.float64)
    y = o.rmsnorm(x, np.full(256, BF16_ONE, np.uint16), 0.0)
    assert abs(np.mean(y.astype(np.float64) ** 2) - 1.0) < 1e-5
    np.testing.assert_allclose(o.rmsnorm(7.0 * x, np.full(256, BF16_ONE, np.uint16), 0.0), y,
                               rtol=1e-5, atol=1e-6)
    # the gain multiplies elementwise
    g = synth.f32_to_bf16(synth.normal_f32(2, 2, 256, 1.0, 0.1))
    np.testing.assert_allclose(o.rmsnorm(x, g, 0.0), y * synth.bf16_to_f32(g), rtol=1e-5,
                               atol=1e-6)


# ---------------------------------------------------------------- RoPE


def test_rope_pairing_and_frequencies():
    o = oracle.Oracle("f64")
    d, base = 8, 10000.0
    for i in range(d // 2):
        for pos in (0, 1, 5, 123):
            v = np.zeros(d)
            v[i] = 1.0
            r = o.rope(v, 1, d, pos, base)
            ang = pos * base ** (-2.0 * i / d)
            want = np.zeros(d)
            want[i] = math.cos(ang)
            want[i + d // 2] = math.sin(ang)
            np.testing.assert_allclose(r, want, atol=1e-12)


def test_rope_d2_is_plane_rotation():
    o = oracle.Oracle("f64")
    for pos in (0, 1, 2, 77):
        r = o.rope(np.array([0.3, -1.2]), 1, 2, pos, 1e6)
        c, s = math.cos(pos), math.sin(pos)
        np.testing.assert_allclose(r, [0.3 * c + 1.2 * s, -1.2 * c + 0.3 * s], atol=1e-12)


@pytest.mark.parametrize("prec,tol", [("f64", 1e-10), ("f32", 2e-4)])
def test_rope_norm_and_relative_position(prec, tol):
    o = oracle.Oracle(prec)
    d, H = 128, 3
    q = synth.normal_f32(9, 1, H * d, 0.0, 1.0).astype(np.float64)
    k = synth.normal_f32(9, 2, H * d, 0.0, 1.0).astype(np.float64)
    for pos in (0, 17, 4095):
        r = o.rope(q, H, d, pos, 1e6).reshape(H, d)
        np.testing.assert_allclose(np.linalg.norm(r, axis=1), np.linalg.norm(q.reshape(H, d), axis=1),
                                   rtol=tol)
    np.testing.assert_array_equal(o.rope(q, H, d, 0, 1e6), q.astype(o.dtype))

    def dot(m, n):
        a = o.rope(q, H, d, m, 1e6).reshape(H, d).astype(np.float64)
        b = o.rope(k, H, d, n, 1e6).reshape(H, d).astype(np.float64)
        return (a * b).sum(axis=1)

    scale = np.abs(q).sum() + np.abs(k).sum()
    for m, n, j in ((5, 2, 100), (0, 0, 31), (1000, 10, 3000)):
        np.testing.assert_allclose(dot(m, n), dot(m + j, n + j), atol=tol * scale)


# ---------------------------------------------------------------- softmax / silu


@pytest.mark.parametrize("prec", ["f32", "f64"])
def test_softmax_properties(prec):
    o = oracle.Oracle(prec)
    s = synth.normal_f32(4, 4, 1000, 0.0, 3.0)
    p = o.softmax(s)
    assert abs(p.astype(np.float64).sum() - 1.0) < 1e-6
    np.testing.assert_allclose(o.softmax(s + 50.0), p, rtol=1e-5, atol=1e-9)
    p2 = o.softmax(np.array([0.7, -0.4]))
    np.testing.assert_allclose(p2[0], 1.0 / (1.0 + math.exp(-1.1)), rtol=1e-6)
    assert int(np.argmax(p)) == int(np.argmax(s))


def test_silu_mul_special_values():
    o = oracle.Oracle("f64")
    g = np.array([0.0, 1.0, 40.0, -40.0, -1.0])
    u = np.array([3.0, 1.0, 2.0, 5.0, 1.0])
    out = o.silu_mul(g, u)
    want = [0.0, 0.7310585786300049, 80.0, 0.0, -0.2689414213699951]
    np.testing.assert_allclose(out, want, atol=1e-12)


def test_argmax_lowest_index_on_ties():
    assert oracle.argmax(np.array([1.0, 3.0, 3.0, 2.0], np.float32)) == 1
    assert oracle.argmax(np.array([-1.0, -1.0], np.float32)) == 0
    assert oracle.argmax(np.array([0.0, 0.0, 0.5], np.float32)) == 2


# ---------------------------------------------------------------- GEMVs


def _dequant_int4(codes, scales_bf16):
    s = synth.bf16_to_f32(scales_bf16).astype(np.float64)
    return codes.astype(np.float64) * np.repeat(s, 128, axis=1)


@pytest.mark.parametrize("prec,rtol", [("f64", 1e-12), ("f32", 1e-5)])
def test_gemv_int4_matches_library_matmul(prec, rtol):
    o = oracle.Oracle(prec)
    N, K = 37, 640
    codes, scales = sm.quantized_tensor(sm.FMT_INT4_G128, 5, 77, N, K)
    x = synth.normal_f32(5, 78, K, 0.0, 1.0).astype(np.float64)
    bias = synth.f32_to_bf16(synth.normal_f32(5, 79, N, 0.0, 0.02))
    y, absacc = o.gemv_int4(oracle.pack_int4(codes), scales, x, bias)
    W = _dequant_int4(codes, scales)
    ref = W @ x + synth.bf16_to_f32(bias)
    bound = rtol * (np.abs(W) @ np.abs(x)) + 1e-12
    assert np.all(np.abs(y - ref) <= bound)
    np.testing.assert_allclose(absacc, np.abs(W) @ np.abs(x), rtol=1e-5)


def test_gemv_int4_single_group_exact():
    # one nonzero group (row 2, group 1), power-of-two scale: result is exact integer arithmetic
    o = oracle.Oracle("f32")
    N, K = 4, 384
    codes = np.zeros((N, K), np.int8)
    grp = np.arange(128) % 16 - 8
    codes[2, 128:256] = grp
    scales = np.full((N, K // 128), 0x3F80, np.uint16)   # 1.0
    scales[2, 1] = 0x3E80                                  # 0.25
    x = np.zeros(K)
    x[128:256] = np.arange(128) % 5 - 2
    y, _ = o.gemv_int4(oracle.pack_int4(codes), scales, x)
    want = np.zeros(N)
    want[2] = 0.25 * float((grp * (np.arange(128) % 5 - 2)).sum())
    np.testing.assert_array_equal(y, want)


def test_gemv_int4_identity_codes():
    o = oracle.Oracle("f32")
    K = 256
    codes = np.eye(K, dtype=np.int8)
    scales = np.full((K, 2), 0x3F80, np.uint16)
    x = synth.normal_f32(6, 6, K, 0.0, 1.0)
    y, _ = o.gemv_int4(oracle.pack_int4(codes), scales, x)
    np.testing.assert_array_equal(y, x)


def test_gemv_int8_and_bf16_match_library_matmul():
    o = oracle.Oracle("f64")
    N, K = 29, 300
    codes, scales = sm.quantized_tensor(sm.FMT_INT8_ROW, 8, 1, N, K)
    x = synth.normal_f32(8, 2, K, 0.0, 1.0).astype(np.float64)
    y, _ = o.gemv_int8(codes, scales, x)
    W = codes.astype(np.float64) * scales.astype(np.float64)[:, None]
    np.testing.assert_allclose(y, W @ x, rtol=1e-12, atol=1e-14)
    w16 = synth.f32_to_bf16(synth.normal_f32(8, 3, N * K, 0.0, 0.02)).reshape(N, K)
    y2, _ = o.gemv_bf16(w16, x)
    np.testing.assert_allclose(y2, synth.bf16_to_f32(w16).astype(np.float64) @ x, rtol=1e-12,
                               atol=1e-14)


# ---------------------------------------------------------------- attention


def _brute_attention(q, kc, vc, Hq, Hkv, d):
    """Direct evaluation on tiny inputs: scores, exponentials, normalised weighted sum."""
    T = kc.shape[0]
    K = synth.bf16_to_f32(kc).astype(np.float64)
    V = synth.bf16_to_f32(vc).astype(np.float64)
    out = np.zeros(Hq * d)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = [sum(q[h * d + i] * K[t, g, i] for i in range(d)) / math.sqrt(d) for t in range(T)]
        e = [math.exp(v - max(s)) for v in s]
        z = sum(e)
        for i in range(d):
            out[h * d + i] = sum(e[t] / z * V[t, g, i] for t in range(T))
    return out


@pytest.mark.parametrize("T,Hq,Hkv,d", [(1, 2, 1, 4), (3, 4, 2, 2), (8, 6, 2, 4), (5, 7, 1, 4)])
def test_attention_brute_force(T, Hq, Hkv, d):
    o = oracle.Oracle("f64")
    q = synth.normal_f32(T, 1, Hq * d, 0.0, 1.0).astype(np.float64)
    kc = synth.f32_to_bf16(synth.normal_f32(T, 2, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    vc = synth.f32_to_bf16(synth.normal_f32(T, 3, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    np.testing.assert_allclose(o.attention(q, kc, vc, Hq, Hkv, d),
                               _brute_attention(q, kc, vc, Hq, Hkv, d), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("ratio", [7, 6, 4, 2])
def test_gqa_equals_replicated_mha(ratio):
    o = oracle.Oracle("f64")
    Hkv, d, T = 2, 16, 33
    Hq = Hkv * ratio
    q = synth.normal_f32(ratio, 1, Hq * d, 0.0, 1.0).astype(np.float64)
    kc = synth.f32_to_bf16(synth.normal_f32(ratio, 2, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    vc = synth.f32_to_bf16(synth.normal_f32(ratio, 3, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    gqa = o.attention(q, kc, vc, Hq, Hkv, d)
    kr = np.repeat(kc, ratio, axis=1)
    vr = np.repeat(vc, ratio, axis=1)
    mha = o.attention(q, kr, vr, Hq, Hq, d)
    np.testing.assert_array_equal(gqa, mha)


def test_attention_degenerate_cases():
    o = oracle.Oracle("f64")
    d = 8
    q = synth.normal_f32(1, 1, 2 * d, 0.0, 1.0).astype(np.float64)
    kc = synth.f32_to_bf16(synth.normal_f32(1, 2, 1 * d, 0.0, 1.0)).reshape(1, 1, d)
    vc = synth.f32_to_bf16(synth.normal_f32(1, 3, 1 * d, 0.0, 1.0)).reshape(1, 1, d)
    # one position: the output is that position's value row for every head
    out = o.attention(q, kc, vc, 2, 1, d).reshape(2, d)
    for h in range(2):
        np.testing.assert_array_equal(out[h], synth.bf16_to_f32(vc[0, 0]))
    # identical keys: uniform weights, output is the mean of V
    T = 5
    kc = np.repeat(kc, T, axis=0)
    vc = synth.f32_to_bf16(synth.normal_f32(1, 4, T * d, 0.0, 1.0)).reshape(T, 1, d)
    out = o.attention(q, kc, vc, 2, 1, d).reshape(2, d)
    np.testing.assert_allclose(out[0], synth.bf16_to_f32(vc[:, 0]).astype(np.float64).mean(0),
                               rtol=1e-12)
