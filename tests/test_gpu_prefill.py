"""Batched prefill on the tensor cores (GPU required).

The prompt runs as GEMMs (weights dequantized to fp16, tcgen05 MMA with fp32 accumulators)
plus causal flash attention.  Checked three ways:
  * the two building blocks through the C ABI: fp16 dequantization (bit-exact: every INT4
    weight is exact in fp16; INT8 rounds once, the same way numpy does) and the GEMM
    against a float64 matmul of the same fp16 operands (fp32 accumulation of K products:
    |err| <= 1e-5 * sum_k |a_mk b_nk| is far above the bound K * 2^-24 for the K here);
  * the whole prompt against the CPU oracle fed token by token, with the engine tests'
    acceptance (max |dlogit| <= 2e-2 * max |logit|, argmax equal where the margin > 5e-2),
    at the tiny shape and at the full widths of the 1.5B, 7B and Qwen3-8B shapes (2 layers);
  * batched against token-by-token prefill on the same engine: logits and the K/V rows
    written to the paged cache.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import model as sm

from ._gpu import device_model, kv_pool_views, to_dev
from .test_gpu_engine import SEED, check_logits, synth_perm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import quantized_decode_gb300 as qd
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return qd.load()


@pytest.mark.parametrize("N,K", [(128, 128), (384, 3584), (1000, 1536)])
def test_dequant_int4_is_exact(lib, N, K):
    import quantized_decode_gb300 as qd
    codes, scales = sm.quantized_tensor(sm.FMT_INT4_G128, 21, N + K, N, K)
    w = to_dev(qd.pack_int4(codes))
    s = to_dev(scales)
    out = torch.empty((N, K), dtype=torch.float16, device="cuda")
    assert lib.llm_op_dequant_f16(1, w.data_ptr(), s.data_ptr(), N, K, out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    # the oracle's own unpacking of the packed words, times the group scale
    unpacked = oracle.unpack_int4(oracle.pack_int4(codes), K).astype(np.float64)
    np.testing.assert_array_equal(unpacked, codes)
    sc = (scales.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = unpacked * np.repeat(sc, 128, axis=1)
    got = out.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, ref)


def test_dequant_int8_rounds_like_numpy(lib):
    N, K = 256, 4096
    codes, scales = sm.quantized_tensor(sm.FMT_INT8_ROW, 22, N + K, N, K)
    w = to_dev(np.ascontiguousarray(codes, np.int8))
    s = to_dev(np.ascontiguousarray(scales, np.float32))
    out = torch.empty((N, K), dtype=torch.float16, device="cuda")
    assert lib.llm_op_dequant_f16(2, w.data_ptr(), s.data_ptr(), N, K, out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    ref = (codes.astype(np.float32) * scales.astype(np.float32)[:, None]).astype(np.float16)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)


def _f16(seed, tid, rows, cols, std):
    return synth.normal_f32(seed, tid, rows * cols, 0.0, std).astype(np.float16).reshape(rows, cols)


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (128, 128, 128), (130, 256, 320), (200, 384, 1024),
                                   (512, 4608, 3584), (77, 3584, 18944)])
def test_gemm_f16_vs_float64(lib, M, N, K):
    a = _f16(31, M * 7 + K, M, K, 1.0)
    b = _f16(32, N * 7 + K, N, K, 0.05)
    ad, bd = to_dev(a), to_dev(b)
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    assert lib.llm_op_gemm_f16(ad.data_ptr(), bd.data_ptr(), M, N, K, c.data_ptr(), None) == 0
    torch.cuda.synchronize()
    got = c.cpu().numpy().astype(np.float64)
    rows = np.arange(M) if M * N * K <= 2 ** 31 else np.arange(0, M, 5)
    a64, b64 = a.astype(np.float64)[rows], b.astype(np.float64)
    ref = a64 @ b64.T
    absacc = np.abs(a64) @ np.abs(b64).T
    err = np.abs(got[rows] - ref)
    assert np.all(err <= 1e-5 * absacc + 1e-30), float(np.max(err / absacc))


@pytest.mark.parametrize("fmt,M,N,K", [(1, 1, 128, 128), (1, 130, 256, 384), (1, 512, 4608, 3584),
                                       (1, 77, 3584, 18944), (2, 200, 384, 4096), (2, 64, 256, 12288),
                                       (1, 600, 384, 512), (1, 1024, 4608, 1024), (2, 300, 1024, 1024),
                                       (1, 512, 37888, 3584)])
def test_gemm_quant_vs_float64(lib, fmt, M, N, K):
    """In-kernel dequantization: C against a float64 matmul of A and the exactly dequantized
    weights (INT4: the oracle's unpacking x the bf16 group scale; INT8: code x fp32 row scale, the
    kernel multiplying the row's fp32 sum of code x activation by the scale)."""
    import quantized_decode_gb300 as qd
    a = _f16(41, M * 7 + K, M, K, 1.0)
    if fmt == 1:
        codes, scales = sm.quantized_tensor(sm.FMT_INT4_G128, 42, N + K, N, K)
        w = to_dev(qd.pack_int4(codes))
        sc = (scales.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        wref = oracle.unpack_int4(oracle.pack_int4(codes), K).astype(np.float64) * np.repeat(sc, 128, axis=1)
    else:
        codes, scales = sm.quantized_tensor(sm.FMT_INT8_ROW, 43, N + K, N, K)
        w = to_dev(np.ascontiguousarray(codes, np.int8))
        wref = codes.astype(np.float64) * scales.astype(np.float32).astype(np.float64)[:, None]
    s = to_dev(scales)
    ad = to_dev(a)
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    assert lib.llm_op_gemm_quant(fmt, ad.data_ptr(), w.data_ptr(), s.data_ptr(), M, N, K, c.data_ptr(), None) == 0
    torch.cuda.synchronize()
    got = c.cpu().numpy().astype(np.float64)
    rows = np.arange(M) if M * N * K <= 2 ** 31 else np.arange(0, M, 5)
    a64 = a.astype(np.float64)[rows]
    ref = a64 @ wref.T
    absacc = np.abs(a64) @ np.abs(wref).T
    err = np.abs(got[rows] - ref)
    assert np.all(err <= 1e-5 * absacc + 1e-30), float(np.max(err / absacc))


def test_gemm_f16_rejects_bad_shapes(lib):
    a = torch.zeros((4, 64), dtype=torch.float16, device="cuda")
    b = torch.zeros((100, 64), dtype=torch.float16, device="cuda")
    c = torch.zeros((4, 100), dtype=torch.float32, device="cuda")
    from quantized_decode_gb300 import _lib as L
    assert lib.llm_op_gemm_f16(a.data_ptr(), b.data_ptr(), 4, 100, 64, c.data_ptr(), None) == L.LLM_ERR_ARG
    assert lib.llm_op_gemm_f16(a.data_ptr(), b.data_ptr(), 4, 128, 60, c.data_ptr(), None) == L.LLM_ERR_ARG


@pytest.fixture(scope="module")
def tiny():
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS["tiny"]
    eng = Engine(device_model(cfg, SEED))
    yield cfg, eng
    eng.set_prefill_batched(True)
    eng.close()


def _oracle_prompt(orc, prompt, pos0=0):
    ref = None
    for i, t in enumerate(prompt):
        ref = orc.step(int(t), pos0 + i)
    return ref


@pytest.mark.parametrize("n", [2, 37, 128, 129, 255])
def test_batched_prefill_vs_oracle_tiny(tiny, n):
    cfg, eng = tiny
    eng.set_prefill_batched(True)
    prompt = sm.prompt(cfg, SEED + n, n)
    eng.reset()
    first = eng.prefill(prompt)
    orc = oracle.OracleModel(cfg, SEED)
    ref = _oracle_prompt(orc, prompt)
    check_logits(eng.logits(), ref, f"prefill n={n}")
    assert first == int(np.argmax(eng.logits()))
    assert eng.seq_len() == n
    if n < cfg.max_context:
        tok = int(np.argmax(ref))
        eng.decode_step(tok)
        check_logits(eng.logits(), orc.step(tok, n), f"decode after prefill n={n}")


def test_prefill_continues_an_existing_sequence(tiny):
    """Two prompts back to back: the second one's rows attend to the first one's cache."""
    cfg, eng = tiny
    eng.set_prefill_batched(True)
    a, b = sm.prompt(cfg, SEED, 40), sm.prompt(cfg, SEED + 9, 30)
    eng.reset()
    eng.prefill(a)
    eng.prefill(b)
    orc = oracle.OracleModel(cfg, SEED)
    _oracle_prompt(orc, a)
    ref = _oracle_prompt(orc, b, 40)
    check_logits(eng.logits(), ref, "second prompt")
    assert eng.seq_len() == 70


def test_batched_equals_token_by_token_prefill(tiny):
    cfg, eng = tiny
    prompt = sm.prompt(cfg, SEED + 3, 97)
    kp, vp, ptv = kv_pool_views(eng, cfg)
    n_pages = ptv.numel()
    ptv.copy_(torch.from_numpy(synth_perm(n_pages)).cuda())
    out = {}
    for batched in (True, False):
        eng.set_prefill_batched(batched)
        kp.zero_()
        vp.zero_()
        eng.reset()
        first = eng.prefill(prompt)
        out[batched] = (first, eng.logits(), kp.clone(), vp.clone())
    eng.set_prefill_batched(True)
    ptv.copy_(torch.arange(n_pages, dtype=torch.int32, device="cuda"))
    (f1, l1, k1, v1), (f0, l0, k0, v0) = out[True], out[False]
    scale = float(np.max(np.abs(l0)))
    assert float(np.max(np.abs(l1 - l0))) <= 2e-2 * scale
    top2 = np.sort(l0)[-2:]
    if top2[1] - top2[0] > 5e-2:
        assert f1 == f0
    for a_, b_ in ((k1, k0), (v1, v0)):
        fa = (a_.cpu().numpy().astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
        fb = (b_.cpu().numpy().astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
        assert np.array_equal(fa == 0, fb == 0)          # the same slots written
        assert float(np.max(np.abs(fa - fb))) <= 2e-2 * float(np.max(np.abs(fb)))


WIDE = [("qwen2.5-7b", 150), ("qwen2.5-1.5b", 131), ("qwen3-8b", 140)]


@pytest.mark.parametrize("name,n", WIDE, ids=[w[0] for w in WIDE])
def test_full_width_prefill_two_layers_vs_oracle(name, n):
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS[name].with_(n_layers=2)
    eng = Engine(device_model(cfg, SEED))
    try:
        prompt = sm.prompt(cfg, SEED, n)
        first = eng.prefill(prompt)
        orc = oracle.OracleModel(cfg, SEED, t_max=n + 4)
        ref = _oracle_prompt(orc, prompt)
        check_logits(eng.logits(), ref, f"{name} prefill")
        assert first == int(np.argmax(eng.logits()))
        tok = int(np.argmax(ref))
        eng.decode_step(tok)
        check_logits(eng.logits(), orc.step(tok, n), f"{name} first decode step")
    finally:
        eng.close()


def test_prompt_longer_than_one_chunk_two_layers_vs_oracle():
    """1100 prompt rows: two prefill chunks (1024 + 76 rows, the second at position 1024 over the
    first chunk's cache), then a decode step; 1.5B widths, 2 layers, against the oracle's own
    prefill (bitwise the same as 1100 oracle steps)."""
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS["qwen2.5-1.5b"].with_(n_layers=2)
    n = 1100
    eng = Engine(device_model(cfg, SEED))
    try:
        prompt = sm.prompt(cfg, SEED + 5, n)
        first = eng.prefill(prompt)
        orc = oracle.OracleModel(cfg, SEED, t_max=n + 4)
        ref = orc.prefill(prompt)
        check_logits(eng.logits(), ref, "1100-row prefill")
        assert first == int(np.argmax(eng.logits()))
        assert eng.seq_len() == n
        tok = int(np.argmax(ref))
        eng.decode_step(tok)
        check_logits(eng.logits(), orc.step(tok, n), "decode after the 1100-row prefill")
    finally:
        eng.close()
