"""The persistent whole-step kernel (GPU required).

Checks it against the CPU oracle at the full widths of the 1.5B, 7B and Qwen3-8B shapes
(two layers each, full vocabulary, seeded K/V written through a shuffled page table), and
against the kernel chain (llm_set_persistent(0)) on the same inputs.  Tolerances are those
of the engine tests: max |GPU - oracle| <= 2e-2 * max |oracle|, argmax equal where the
oracle's top-1/top-2 margin exceeds 5e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import model as sm

from ._gpu import device_model, fill_kv
from .test_gpu_engine import SEED, check_logits, synth_perm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    from quantized_decode_gb300 import Engine
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    cfg = sm.CONFIGS["tiny"]
    eng = Engine(device_model(cfg, SEED))
    yield cfg, eng
    eng.close()


def _forced(eng, prompt, forced):
    eng.reset()
    eng.prefill(prompt)
    out = [eng.logits()]
    for t in forced:
        eng.decode_step(int(t))
        out.append(eng.logits())
    return out


def test_persistent_matches_chain_and_oracle_tiny(tiny):
    cfg, eng = tiny
    prompt = sm.prompt(cfg, SEED, 24)
    forced = sm.prompt(cfg, SEED + 1, 10)
    runs = {}
    for mode in (True, False):
        eng.set_persistent(mode)
        runs[mode] = _forced(eng, prompt, forced)
    eng.set_persistent(True)
    orc = oracle.OracleModel(cfg, SEED)
    ref = None
    for pos, t in enumerate(prompt):
        ref = orc.step(int(t), pos)
    refs = [ref] + [orc.step(int(t), len(prompt) + i) for i, t in enumerate(forced)]
    for i, r in enumerate(refs):
        check_logits(runs[True][i], r, f"persistent step {i}")
        check_logits(runs[False][i], r, f"chain step {i}")
        scale = float(np.max(np.abs(r)))
        assert float(np.max(np.abs(runs[True][i] - runs[False][i]))) <= 2e-2 * scale


def test_persistent_profile_regions(tiny):
    cfg, eng = tiny
    eng.set_persistent(True)
    eng.reset()
    eng.prefill(sm.prompt(cfg, SEED, 8))
    ms = eng.profile_step()
    assert ms.shape == (5 * cfg.n_layers + 1,)
    assert np.all(ms >= 0) and float(ms.sum()) > 0
    assert eng.seq_len() == 9


def test_persistent_repeat_is_bitwise(tiny):
    """Counters reset themselves: the same steps give the same bits every time."""
    cfg, eng = tiny
    eng.set_persistent(True)
    prompt = sm.prompt(cfg, SEED, 30)
    a = _forced(eng, prompt, [5, 6, 7])
    b = _forced(eng, prompt, [5, 6, 7])
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


# Full-width shapes, two layers each: (name, cached tokens before the forced steps)
WIDE = [("qwen2.5-7b", 1000), ("qwen2.5-1.5b", 333), ("qwen3-8b", 1500)]


@pytest.mark.parametrize("name,T0", WIDE, ids=[w[0] for w in WIDE])
def test_full_width_two_layers_vs_oracle(name, T0):
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS[name].with_(n_layers=2)
    eng = Engine(device_model(cfg, SEED))
    try:
        eng.set_persistent(True)                       # raises if the shape were unsupported
        n_pages = (cfg.max_context + 15) // 16
        ks, vs = fill_kv(eng, cfg, 11, T0, page_perm=synth_perm(n_pages))
        orc = oracle.OracleModel(cfg, SEED)
        for l in range(cfg.n_layers):
            orc.set_kv(l, ks[l], vs[l])
        tok = 7
        logits = []
        for i in range(3):
            got = eng.decode_step(tok)
            ref = orc.step(tok, T0 + i)
            check_logits(eng.logits(), ref, f"{name} step {i}")
            assert got == int(np.argmax(eng.logits()))
            logits.append(eng.logits())
            tok = int(np.argmax(ref))
        # the kernel chain on the same cache and tokens
        eng.set_persistent(False)
        eng.debug_kv(set_len=T0)
        tok = 7
        ref_orc = oracle.OracleModel(cfg, SEED)
        for l in range(cfg.n_layers):
            ref_orc.set_kv(l, ks[l], vs[l])
        for i in range(3):
            eng.decode_step(tok)
            ref = ref_orc.step(tok, T0 + i)
            check_logits(eng.logits(), ref, f"{name} chain step {i}")
            scale = float(np.max(np.abs(ref)))
            assert float(np.max(np.abs(eng.logits() - logits[i]))) <= 2e-2 * scale
            tok = int(np.argmax(ref))
    finally:
        eng.close()


def test_full_width_steps_do_not_stall():
    """Every wait in the kernel is bounded by 1 s; a step that finishes only through such a
    timeout (a wait on the wrong barrier phase) is still correct but takes ~1 s.  Twenty steps
    of the 2-layer 7B shape take well under a millisecond each."""
    import time
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS["qwen2.5-7b"].with_(n_layers=2)
    eng = Engine(device_model(cfg, SEED))
    try:
        eng.set_persistent(True)
        fill_kv(eng, cfg, 11, 3000)
        eng.decode_step(7)
        t0 = time.perf_counter()
        for _ in range(20):
            eng.decode_step()
        assert time.perf_counter() - t0 < 0.5
    finally:
        eng.close()


def test_counter_wait_that_runs_out_returns_timeout_and_reset_recovers(tiny):
    """The failure path of a bounded device wait, without any GPU fault: the test hook makes
    the persistent kernel's phase-counter waits expect one arrival more than will come, with
    a 2 ms bound.  The step must come back with LLM_ERR_TIMEOUT well within a second (the
    kernel records the timeout, stops issuing copies, drains the ones in flight and
    returns), and after llm_reset the engine must reproduce a clean run bit for bit."""
    import ctypes
    import time
    from quantized_decode_gb300 import _lib as L
    cfg, eng = tiny
    eng.set_persistent(True)
    prompt = sm.prompt(cfg, SEED, 12)
    want = _forced(eng, prompt, [5, 6, 7])
    eng.reset()
    eng.prefill(prompt)
    eng.debug_step_wait(1, 2_000_000)
    try:
        out = ctypes.c_int32()
        for _ in range(2):                 # the sticky word keeps reporting until llm_reset
            t0 = time.perf_counter()
            rc = eng.lib.llm_decode_step(eng.h, 5, ctypes.byref(out))
            dt = time.perf_counter() - t0
            assert rc == L.LLM_ERR_TIMEOUT, rc
            assert dt < 0.5, dt
    finally:
        eng.debug_step_wait(0, 1_000_000_000)
    eng.reset()
    got = _forced(eng, prompt, [5, 6, 7])
    for x, y in zip(want, got):
        np.testing.assert_array_equal(x, y)
    eng.set_persistent(False)
