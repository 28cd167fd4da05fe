"""Single kernels through the C ABI (llm_ops.h) against the CPU oracle (GPU required).

Tolerance for the dequant GEMVs, derived from the kernel's arithmetic: activations are
rounded once to fp16 (relative 2^-11), each code*activation product is rounded to fp16
(2^-11), and products are summed in fp16 chains of at most 8 before widening to fp32
(at most 8 roundings of 2^-11 relative to the chain's |sum|).  Per output that bounds the
error by (2 + 8) * 2^-11 * sum_k |W_nk x_k| < 5e-3 * absacc; tests use 6e-3 * absacc.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import model as sm

from ._gpu import to_dev

pytestmark = pytest.mark.gpu

GEMV_TOL = 6e-3


@pytest.fixture(scope="module")
def lib():
    import quantized_decode_gb300 as qd
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return qd.load()


def _gemv_int4(lib, codes, scales, x, bias=None):
    import quantized_decode_gb300 as qd
    N, K = codes.shape
    w = to_dev(qd.pack_int4(codes))
    s = to_dev(scales)
    b = to_dev(bias) if bias is not None else None
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    rc = lib.llm_op_gemv_int4(w.data_ptr(), s.data_ptr(), b.data_ptr() if b is not None else None,
                              N, K, xd.data_ptr(), y.data_ptr(), None)
    assert rc == 0
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("N,K", [(32, 256), (64, 768), (128, 1536), (4608, 3584), (3584, 18944),
                                 (96, 8960), (256, 4096), (512, 12288)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_gemv_int4_vs_oracle(lib, N, K, with_bias):
    codes, scales = sm.quantized_tensor(sm.FMT_INT4_G128, 11, N + K, N, K)
    x = synth.normal_f32(12, K, K, 0.0, 1.0)
    bias = synth.f32_to_bf16(synth.normal_f32(13, N, N, 0.0, 0.02)) if with_bias else None
    y = _gemv_int4(lib, codes, scales, x, bias)
    ref, absacc = oracle.Oracle("f64").gemv_int4(oracle.pack_int4(codes), scales, x, bias)
    err = np.abs(y - ref)
    assert np.all(err <= GEMV_TOL * absacc + 1e-6), float(np.max(err / (absacc + 1e-30)))
    # typical error is far below the worst-case bound
    assert np.sqrt(np.mean(err ** 2)) <= 1e-3 * np.sqrt(np.mean(ref ** 2))


def test_gemv_int4_extreme_activation_range(lib):
    N, K = 64, 1024
    codes, scales = sm.quantized_tensor(sm.FMT_INT4_G128, 5, 1, N, K)
    x = synth.normal_f32(6, 1, K, 0.0, 1.0)
    x[::7] *= 3e4          # large entries would overflow fp16 without the power-of-two prescale
    x[1::7] *= 1e-5
    y = _gemv_int4(lib, codes, scales, x)
    ref, absacc = oracle.Oracle("f64").gemv_int4(oracle.pack_int4(codes), scales, x)
    assert np.all(np.isfinite(y))
    assert np.all(np.abs(y - ref) <= GEMV_TOL * absacc + 1e-6)


def test_gemv_int4_zero_input_and_extreme_codes(lib):
    N, K = 32, 256
    codes = np.full((N, K), -8, np.int8)
    codes[::2] = 7
    scales = np.full((N, K // 128), 0x3F80, np.uint16)  # 1.0
    bias = synth.f32_to_bf16(synth.normal_f32(1, 1, N, 0.0, 1.0))
    y0 = _gemv_int4(lib, codes, scales, np.zeros(K, np.float32), bias)
    np.testing.assert_array_equal(y0, synth.bf16_to_f32(bias))
    x = np.ones(K, np.float32)
    y = _gemv_int4(lib, codes, scales, x)
    np.testing.assert_array_equal(y, np.where(np.arange(N) % 2 == 0, 7.0 * K, -8.0 * K))


@pytest.mark.parametrize("N,K", [(32, 256), (256, 4096), (128, 12288), (4096, 4096)])
def test_gemv_int8_vs_oracle(lib, N, K):
    import quantized_decode_gb300 as qd
    codes, scales = sm.quantized_tensor(sm.FMT_INT8_ROW, 21, N + K, N, K)
    x = synth.normal_f32(22, K, K, 0.0, 1.0)
    w, s = to_dev(qd.pack_int8(codes)), to_dev(scales)
    xd = torch.from_numpy(x).cuda()
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    assert lib.llm_op_gemv_int8(w.data_ptr(), s.data_ptr(), N, K, xd.data_ptr(), y.data_ptr(), None) == 0
    torch.cuda.synchronize()
    ref, absacc = oracle.Oracle("f64").gemv_int8(codes, scales, x)
    err = np.abs(y.cpu().numpy() - ref)
    # INT8 chains hold 4 products (|code| <= 127): same bound structure as INT4
    assert np.all(err <= GEMV_TOL * absacc + 1e-6)


def _lm_head(lib, w_dev, scale_dev, gamma, x, N, K, eps=1e-6):
    g = to_dev(gamma)
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    logits = torch.empty(N, dtype=torch.float32, device="cuda")
    tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = lib.llm_op_lm_head_argmax(w_dev.data_ptr(), scale_dev.data_ptr() if scale_dev is not None else None,
                                   g.data_ptr(), eps, N, K, xd.data_ptr(), logits.data_ptr(),
                                   tok.data_ptr(), None)
    assert rc == 0
    torch.cuda.synchronize()
    return logits.cpu().numpy(), int(tok.item())


@pytest.mark.parametrize("N,K", [(1024, 256), (151936, 1536), (152064, 3584)])
def test_lm_head_bf16_vs_oracle(lib, N, K):
    w = synth.f32_to_bf16(synth.normal_f32(31, N, N * K, 0.0, 0.02)).reshape(N, K)
    gamma = synth.f32_to_bf16(synth.normal_f32(32, K, K, 1.0, 0.01))
    x = synth.normal_f32(33, K, K, 0.0, 3.0)
    logits, tok = _lm_head(lib, to_dev(w), None, gamma, x, N, K)
    o = oracle.Oracle("f64")
    n = o.rmsnorm(x, gamma, 1e-6)
    ref, absacc = o.gemv_bf16(w, n)
    assert np.all(np.abs(logits - ref) <= 1e-5 * absacc + 1e-6)
    assert tok == int(np.argmax(logits))           # the kernel's own argmax is exact
    srt = np.sort(ref)
    if srt[-1] - srt[-2] > 1e-3:
        assert tok == int(np.argmax(ref))


def test_lm_head_ties_pick_lowest_index(lib):
    N, K = 4096, 256
    w = synth.f32_to_bf16(synth.normal_f32(41, 1, N * K, 0.0, 0.02)).reshape(N, K)
    w[3001] = w[17]                 # identical rows -> identical logits
    w[17] = synth.f32_to_bf16(np.full(K, 0.05, np.float32))
    w[3001] = w[17]
    w[4000] = w[17]
    gamma = np.full(K, 0x3F80, np.uint16)
    x = np.ones(K, np.float32)
    logits, tok = _lm_head(lib, to_dev(w), None, gamma, x, N, K)
    assert logits[17] == logits[3001] == logits[4000]
    assert tok == 17


def test_lm_head_int8_vs_oracle(lib):
    import quantized_decode_gb300 as qd
    N, K = 151936, 4096
    codes, scales = sm.quantized_tensor(sm.FMT_INT8_ROW, 51, 2, N, K)
    gamma = synth.f32_to_bf16(synth.normal_f32(52, K, K, 1.0, 0.01))
    x = synth.normal_f32(53, K, K, 0.0, 2.0)
    logits, tok = _lm_head(lib, to_dev(qd.pack_int8(codes)), to_dev(scales), gamma, x, N, K)
    o = oracle.Oracle("f64")
    ref, absacc = o.gemv_int8(codes, scales, o.rmsnorm(x, gamma, 1e-6))
    assert np.all(np.abs(logits - ref) <= GEMV_TOL * absacc + 1e-6)
    assert tok == int(np.argmax(logits))


# ---------------------------------------------------------------- attention


def _paged(kc, vc, n_pages_total, perm):
    """Contiguous bf16 [T][Hkv][d] -> pools [pages][Hkv][16][d] placed through perm."""
    T, Hkv, d = kc.shape
    n_pg = (T + 15) // 16
    kp = np.zeros((n_pages_total, Hkv, 16, d), np.uint16)
    vp = np.zeros_like(kp)
    kpad = np.zeros((n_pg * 16, Hkv, d), np.uint16)
    vpad = np.zeros_like(kpad)
    kpad[:T], vpad[:T] = kc, vc
    kp[perm[:n_pg]] = kpad.reshape(n_pg, 16, Hkv, d).transpose(0, 2, 1, 3)
    vp[perm[:n_pg]] = vpad.reshape(n_pg, 16, Hkv, d).transpose(0, 2, 1, 3)
    return kp, vp


def _attention(lib, q, kp, vp, table, T, Hq, Hkv, d, P):
    qd_ = torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda()
    kd, vd, td = to_dev(kp), to_dev(vp), to_dev(np.ascontiguousarray(table, np.int32))
    out = torch.empty(Hq * d, dtype=torch.float32, device="cuda")
    rc = lib.llm_op_attention(qd_.data_ptr(), kd.data_ptr(), vd.data_ptr(), td.data_ptr(),
                              kp.shape[0], T, Hq, Hkv, d, P, out.data_ptr(), None)
    assert rc == 0
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("T", [1, 15, 16, 17, 49, 100, 1000, 4096])
@pytest.mark.parametrize("Hq,Hkv,d", [(4, 2, 64), (28, 4, 128), (12, 2, 128), (32, 8, 128)])
def test_attention_vs_oracle_shuffled_pages(lib, T, Hq, Hkv, d):
    n_pg = (T + 15) // 16
    total = n_pg + 5
    perm = synth.permutation(T, Hq, total)
    q = synth.normal_f32(T, 1, Hq * d, 0.0, 1.0)
    kc = synth.f32_to_bf16(synth.normal_f32(T, 2, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    vc = synth.f32_to_bf16(synth.normal_f32(T, 3, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    kp, vp = _paged(kc, vc, total, perm)
    ref = oracle.Oracle("f64").attention(q, kc, vc, Hq, Hkv, d)
    for P in (1, 3, 0):
        out = _attention(lib, q, kp, vp, perm, T, Hq, Hkv, d, P)
        np.testing.assert_allclose(out, ref, rtol=0, atol=2e-5 * np.max(np.abs(ref)) + 1e-6)


def test_attention_page_table_indirection_is_bit_exact(lib):
    T, Hq, Hkv, d = 777, 28, 4, 128
    n_pg = (T + 15) // 16
    q = synth.normal_f32(7, 1, Hq * d, 0.0, 1.0)
    kc = synth.f32_to_bf16(synth.normal_f32(7, 2, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    vc = synth.f32_to_bf16(synth.normal_f32(7, 3, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    ident = np.arange(n_pg, dtype=np.int32)
    perm = synth.permutation(7, 4, n_pg)
    a = _attention(lib, q, *_paged(kc, vc, n_pg, ident), ident, T, Hq, Hkv, d, 8)
    b = _attention(lib, q, *_paged(kc, vc, n_pg, perm), perm, T, Hq, Hkv, d, 8)
    np.testing.assert_array_equal(a, b)


def test_attention_split_count_invariance(lib):
    T, Hq, Hkv, d = 2000, 28, 4, 128
    n_pg = (T + 15) // 16
    ident = np.arange(n_pg, dtype=np.int32)
    q = synth.normal_f32(8, 1, Hq * d, 0.0, 1.0)
    kc = synth.f32_to_bf16(synth.normal_f32(8, 2, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    vc = synth.f32_to_bf16(synth.normal_f32(8, 3, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    kp, vp = _paged(kc, vc, n_pg, ident)
    base = _attention(lib, q, kp, vp, ident, T, Hq, Hkv, d, 1)
    for P in (2, 16, 125, 200):
        out = _attention(lib, q, kp, vp, ident, T, Hq, Hkv, d, P)
        np.testing.assert_allclose(out, base, rtol=0, atol=1e-5 * np.max(np.abs(base)))


def test_attention_reports_a_page_outside_the_pools(lib):
    """A table entry past the caller's pools is never fetched (page 0 stands in on the
    device) and the call returns LLM_ERR_DEVICE; the next good call returns LLM_OK."""
    from quantized_decode_gb300 import _lib as L
    T, Hq, Hkv, d = 100, 28, 4, 128
    n_pg = (T + 15) // 16
    ident = np.arange(n_pg, dtype=np.int32)
    q = synth.normal_f32(9, 1, Hq * d, 0.0, 1.0)
    kc = synth.f32_to_bf16(synth.normal_f32(9, 2, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    vc = synth.f32_to_bf16(synth.normal_f32(9, 3, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    kp, vp = _paged(kc, vc, n_pg, ident)
    kd, vd = to_dev(kp), to_dev(vp)
    qd_ = torch.from_numpy(q).cuda()
    out = torch.empty(Hq * d, dtype=torch.float32, device="cuda")
    for bad in (n_pg, -1, 1 << 20):
        table = ident.copy()
        table[3] = bad
        td = to_dev(table)
        rc = lib.llm_op_attention(qd_.data_ptr(), kd.data_ptr(), vd.data_ptr(), td.data_ptr(), n_pg,
                                  T, Hq, Hkv, d, 0, out.data_ptr(), None)
        assert rc == L.LLM_ERR_DEVICE, bad
    td = to_dev(ident)
    rc = lib.llm_op_attention(qd_.data_ptr(), kd.data_ptr(), vd.data_ptr(), td.data_ptr(), n_pg, T,
                              Hq, Hkv, d, 0, out.data_ptr(), None)
    assert rc == 0
    # pool extent refused on the host before any launch
    for n_pool in (0, -5, (1 << 31) // (16 * Hkv) + 1):
        rc = lib.llm_op_attention(qd_.data_ptr(), kd.data_ptr(), vd.data_ptr(), td.data_ptr(), n_pool,
                                  T, Hq, Hkv, d, 0, out.data_ptr(), None)
        assert rc == L.LLM_ERR_ARG, n_pool
