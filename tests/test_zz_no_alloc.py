"""The attention entry point that allocates no device memory (GPU required).

Callers that may not allocate device memory when they call in (a host framework owning
all device memory through its own pool, latency-critical paths) use
llm_op_attention_noalloc, whose scratch is a fixed array inside the library.  This file
sorts last so that a run stopping at the first failure has already run every other test;
it sets up everything it uses, so it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth

from ._gpu import to_dev

pytestmark = pytest.mark.gpu


def _case(seed, T, Hq, Hkv, d):
    n_pg = (T + 15) // 16
    perm = synth.permutation(seed, 1, n_pg + 3)
    q = synth.normal_f32(seed, 2, Hq * d, 0.0, 1.0)
    kc = synth.f32_to_bf16(synth.normal_f32(seed, 3, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    vc = synth.f32_to_bf16(synth.normal_f32(seed, 4, T * Hkv * d, 0.0, 1.0)).reshape(T, Hkv, d)
    kp = np.zeros((n_pg + 3, Hkv, 16, d), np.uint16)
    vp = np.zeros_like(kp)
    kpad = np.zeros((n_pg * 16, Hkv, d), np.uint16)
    vpad = np.zeros_like(kpad)
    kpad[:T], vpad[:T] = kc, vc
    kp[perm[:n_pg]] = kpad.reshape(n_pg, 16, Hkv, d).transpose(0, 2, 1, 3)
    vp[perm[:n_pg]] = vpad.reshape(n_pg, 16, Hkv, d).transpose(0, 2, 1, 3)
    return (torch.from_numpy(q).cuda(), to_dev(kp), to_dev(vp), to_dev(perm), n_pg + 3)


def _run(fn, case, T, Hq, Hkv, d, P):
    q, kp, vp, pt, n_pool = case
    out = torch.full((Hq * d,), float("nan"), dtype=torch.float32, device="cuda")
    rc = fn(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), pt.data_ptr(), n_pool, T, Hq, Hkv, d, P,
            out.data_ptr(), None)
    assert rc == 0
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_noalloc_attention_matches_allocating_entry_twice_in_a_row():
    import quantized_decode_gb300 as qd
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    lib = qd.load()
    # two calls in a row on different shapes: the shared array keeps the last call's
    # contents, so the second call must reset what has to start at zero
    for seed, (T, Hq, Hkv, d, P) in ((1, (4096, 28, 4, 128, 0)), (2, (777, 12, 2, 128, 5))):
        case = _case(seed, T, Hq, Hkv, d)
        ref = _run(lib.llm_op_attention, case, T, Hq, Hkv, d, P)
        got = _run(lib.llm_op_attention_noalloc, case, T, Hq, Hkv, d, P)
        np.testing.assert_allclose(got, ref, rtol=0, atol=2e-5 * np.max(np.abs(ref)) + 1e-6)


def test_noalloc_attention_rejects_requests_beyond_its_array():
    import quantized_decode_gb300 as qd
    from quantized_decode_gb300 import _lib as L
    lib = qd.load()
    T, Hq, Hkv, d, P = 64, 64, 8, 128, 256   # 64 * 256 * 130 * 4 bytes > 4 MiB
    case = _case(3, T, 64, Hkv, d)
    q, kp, vp, pt, n_pool = case
    out = torch.zeros(Hq * d, dtype=torch.float32, device="cuda")
    rc = lib.llm_op_attention_noalloc(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), pt.data_ptr(), n_pool,
                                      T, Hq, Hkv, d, P, out.data_ptr(), None)
    assert rc == L.LLM_ERR_ARG


def test_noalloc_attention_reports_a_page_outside_the_pools():
    """The shared array carries the error word too: a bad page returns LLM_ERR_DEVICE and
    the next call (which clears the word) returns LLM_OK with the allocating entry's result."""
    import quantized_decode_gb300 as qd
    from quantized_decode_gb300 import _lib as L
    lib = qd.load()
    T, Hq, Hkv, d = 200, 28, 4, 128
    q, kp, vp, pt, n_pool = _case(4, T, Hq, Hkv, d)
    bad = pt.clone()
    bad[0:4] = torch.tensor([n_pool, 0, 0, 0], dtype=torch.uint8)   # entry 0 := n_pool (past the pools)
    out = torch.zeros(Hq * d, dtype=torch.float32, device="cuda")
    rc = lib.llm_op_attention_noalloc(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), bad.data_ptr(), n_pool,
                                      T, Hq, Hkv, d, 0, out.data_ptr(), None)
    assert rc == L.LLM_ERR_DEVICE
    ref = _run(lib.llm_op_attention, (q, kp, vp, pt, n_pool), T, Hq, Hkv, d, 0)
    got = _run(lib.llm_op_attention_noalloc, (q, kp, vp, pt, n_pool), T, Hq, Hkv, d, 0)
    np.testing.assert_allclose(got, ref, rtol=0, atol=2e-5 * np.max(np.abs(ref)) + 1e-6)
