"""The whole decode step through the C ABI (llm.h) against the CPU oracle (GPU required).

Acceptance (teacher forcing: both sides consume the same tokens):
  max |GPU logits - oracle logits| <= 2e-2 * max |oracle logits|  per step, and
  argmax equal on every step whose oracle top-1/top-2 margin exceeds 5e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import model as sm

from ._gpu import device_model, fill_kv, kv_pool_views

pytestmark = pytest.mark.gpu

SEED = 2024
LOGIT_TOL = 2e-2
MARGIN = 5e-2


def check_logits(gpu, ref, where=""):
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(gpu - ref)))
    assert err <= LOGIT_TOL * scale, f"{where}: max err {err} vs scale {scale}"
    top2 = np.sort(ref)[-2:]
    if top2[1] - top2[0] > MARGIN:
        assert int(np.argmax(gpu)) == int(np.argmax(ref)), where
    return err / scale


@pytest.fixture(scope="module")
def tiny():
    from quantized_decode_gb300 import Engine
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    cfg = sm.CONFIGS["tiny"]
    model = device_model(cfg, SEED)
    eng = Engine(model)
    yield cfg, model, eng
    eng.close()


def _teacher_forced(cfg, eng, orc, n_prompt, n_decode):
    """Prefill a seeded prompt, then decode with the oracle's greedy tokens fed to both."""
    prompt = sm.prompt(cfg, SEED, n_prompt)
    eng.reset()
    first = eng.prefill(prompt)
    ref = None
    for pos, t in enumerate(prompt):
        ref = orc.step(int(t), pos)
    errs = [check_logits(eng.logits(), ref, "prefill")]
    assert first == int(np.argmax(eng.logits()))
    tok = int(np.argmax(ref))
    for i in range(n_decode):
        pos = n_prompt + i
        got = eng.decode_step(tok)
        ref = orc.step(tok, pos)
        errs.append(check_logits(eng.logits(), ref, f"step {i}"))
        assert got == int(np.argmax(eng.logits()))
        tok = int(np.argmax(ref))
    return errs


def test_tiny_prefill_and_decode_vs_oracle(tiny):
    cfg, model, eng = tiny
    orc = oracle.OracleModel(cfg, SEED)
    errs = _teacher_forced(cfg, eng, orc, 64, 16)
    assert max(errs) < LOGIT_TOL


def test_tiny_kv_cache_matches_oracle(tiny):
    cfg, model, eng = tiny
    orc = oracle.OracleModel(cfg, SEED)
    kp, vp, ptv = kv_pool_views(eng, cfg)
    kp.zero_()                                # earlier tests on this engine left rows behind
    vp.zero_()
    _teacher_forced(cfg, eng, orc, 40, 9)
    T = 49                                    # the last page holds one token
    table = ptv.cpu().numpy()
    for pool, ref in ((kp, orc.k_cache), (vp, orc.v_cache)):
        arr = pool.cpu().numpy().view(np.uint16)       # [L][pages][Hkv][16][d]
        got = np.stack([arr[:, table[p // 16], :, p % 16, :] for p in range(T)], axis=1)
        g = (got.astype(np.uint32) << 16).view(np.float32)
        r = (ref[:, :T].astype(np.uint32) << 16).view(np.float32)
        assert np.max(np.abs(g - r)) <= 2e-2 * np.max(np.abs(r))
        # slots past the sequence were never written
        last_page = table[(T - 1) // 16]
        assert np.all(arr[:, last_page, :, T % 16:, :] == 0)


def test_graph_replay_equals_eager_launches(tiny):
    cfg, model, eng = tiny
    prompt = sm.prompt(cfg, SEED, 20)
    outs = []
    for graph in (True, False):
        eng.set_graph_mode(graph)
        eng.reset()
        toks = [eng.prefill(prompt)]
        for _ in range(6):
            toks.append(eng.decode_step())
        outs.append((toks, eng.logits()))
    eng.set_graph_mode(True)
    assert outs[0][0] == outs[1][0]
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_reset_reproduces_bitwise(tiny):
    cfg, model, eng = tiny
    prompt = sm.prompt(cfg, SEED, 33)
    runs = []
    for _ in range(2):
        eng.reset()
        toks = [eng.prefill(prompt)] + [eng.decode_step() for _ in range(5)]
        runs.append((toks, eng.logits()))
    assert runs[0][0] == runs[1][0]
    np.testing.assert_array_equal(runs[0][1], runs[1][1])


def test_enqueue_matches_synchronous_greedy(tiny):
    cfg, model, eng = tiny
    prompt = sm.prompt(cfg, SEED, 10)
    eng.reset()
    eng.prefill(prompt)
    sync_toks = [eng.decode_step() for _ in range(8)]
    eng.reset()
    eng.prefill(prompt)
    eng.decode_enqueue(8)
    eng.sync()
    assert eng.last_token() == sync_toks[-1]
    assert eng.seq_len() == 18


def test_context_full_and_state_errors(tiny):
    from quantized_decode_gb300 import LLMError, _lib as L
    cfg, model, eng = tiny
    eng.reset()
    with pytest.raises(LLMError) as e:
        eng.decode_step()                       # nothing to feed yet
    assert e.value.code == L.LLM_ERR_STATE
    with pytest.raises(LLMError) as e:
        eng.prefill(np.zeros(cfg.max_context + 1, np.int32))
    assert e.value.code == L.LLM_ERR_CONTEXT_FULL
    with pytest.raises(LLMError) as e:
        eng.prefill(np.array([cfg.vocab], np.int32))
    assert e.value.code == L.LLM_ERR_ARG
    eng.prefill(sm.prompt(cfg, SEED, cfg.max_context - 1))
    eng.decode_step()                           # fills the last slot
    with pytest.raises(LLMError) as e:
        eng.decode_step()
    assert e.value.code == L.LLM_ERR_CONTEXT_FULL
    eng.reset()


def test_shuffled_page_table_is_bit_exact(tiny):
    """Same sequence with identity vs shuffled page tables: identical logits, and every K/V
    row lands at slot pos % 16 of page table[pos / 16] with all other slots untouched."""
    cfg, model, eng = tiny
    prompt = sm.prompt(cfg, SEED, 37)
    kp, vp, ptv = kv_pool_views(eng, cfg)
    n_pages = ptv.numel()
    results = []
    for perm in (np.arange(n_pages, dtype=np.int32), synth_perm(n_pages)):
        kp.zero_()
        vp.zero_()
        ptv.copy_(torch.from_numpy(perm).cuda())
        eng.reset()
        toks = [eng.prefill(prompt)] + [eng.decode_step() for _ in range(4)]
        T = 37 + 4
        arr = kp.cpu().numpy()
        rows = np.stack([arr[:, perm[p // 16], :, p % 16, :] for p in range(T)], axis=1)
        written = np.zeros(arr.shape[:4], bool)
        for p in range(T):
            written[:, perm[p // 16], :, p % 16] = True
        assert np.all(arr[~written] == 0)
        results.append((toks, eng.logits(), rows))
    ptv.copy_(torch.arange(n_pages, dtype=torch.int32, device="cuda"))
    assert results[0][0] == results[1][0]
    np.testing.assert_array_equal(results[0][1], results[1][1])
    np.testing.assert_array_equal(results[0][2], results[1][2])


def synth_perm(n):
    import synth
    return synth.permutation(77, 5, n)


def test_seeded_kv_fill_then_decode_vs_oracle(tiny):
    """The long-context protocol on the tiny shape: KV filled with N(0,1) values through a
    shuffled table, then teacher-forced decode steps."""
    cfg, model, eng = tiny
    T0 = 200
    eng.reset()
    ks, vs = fill_kv(eng, cfg, 5, T0, page_perm=synth_perm((cfg.max_context + 15) // 16))
    orc = oracle.OracleModel(cfg, SEED)
    for l in range(cfg.n_layers):
        orc.set_kv(l, ks[l], vs[l])
    tok = 3
    for i in range(8):
        got = eng.decode_step(tok)
        ref = orc.step(tok, T0 + i)
        check_logits(eng.logits(), ref, f"step {i}")
        tok = int(np.argmax(ref))
    kp, vp, ptv = kv_pool_views(eng, cfg)
    ptv.copy_(torch.arange(ptv.numel(), dtype=torch.int32, device="cuda"))
    eng.reset()
