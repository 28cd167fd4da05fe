"""Multi-sequence decode (llm_batch_*) against independent oracle runs (GPU required).

Each sequence of a batch must behave as if it ran alone: its logits after every step meet
the acceptance rule against its own oracle run (max |GPU - oracle| <= 2e-2 max |oracle|,
argmax equal where the oracle's top-1/top-2 margin > 5e-2), whatever the other sequences
do.  The pool's pages are handed out in a shuffled order, sequences have different lengths,
and the K/V rows a sequence wrote are found at slot pos % 16 of its page pos / 16.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import model as sm

from ._gpu import device_model
from .test_gpu_engine import SEED, check_logits

pytestmark = pytest.mark.gpu


def _oracle_prefix(cfg, prompt, t_max):
    orc = oracle.OracleModel(cfg, SEED, t_max=t_max)
    ref = None
    for pos, t in enumerate(prompt):
        ref = orc.step(int(t), pos)
    return orc, ref


def _run_batch(cfg, model, n_seq, max_seqs=8, n_steps=6, lens=None, page_seed=3):
    from quantized_decode_gb300 import BatchEngine
    eng = BatchEngine(model, max_seqs)
    try:
        n_pages = (cfg.max_context + 15) // 16 * max_seqs + 1
        eng.set_page_order(1 + synth.permutation(page_seed, 7, n_pages - 1))
        lens = lens or [5 + 7 * i for i in range(n_seq)]
        seqs, orcs, refs, errs = [], [], [], []
        for i in range(n_seq):
            s = eng.add()
            prompt = sm.prompt(cfg, SEED + i, lens[i], stream=i)
            first = eng.prefill(s, prompt)
            orc, ref = _oracle_prefix(cfg, prompt, cfg.max_context)
            errs.append(check_logits(eng.logits(s), ref, f"seq {i} prefill"))
            assert first == int(np.argmax(eng.logits(s)))
            seqs.append(s)
            orcs.append(orc)
            refs.append(ref)
        for step in range(n_steps):
            toks = [int(np.argmax(r)) for r in refs]
            out = eng.step(seqs, toks)
            for i, s in enumerate(seqs):
                refs[i] = orcs[i].step(toks[i], lens[i] + step)
                got = eng.logits(s)
                errs.append(check_logits(got, refs[i], f"seq {i} step {step}"))
                assert out[i] == int(np.argmax(got))
        return eng, seqs, orcs, lens, max(errs)
    except Exception:
        eng.close()
        raise


@pytest.fixture(scope="module")
def tiny_model():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    cfg = sm.CONFIGS["tiny"].with_(max_context=128)
    return cfg, device_model(cfg, SEED)


@pytest.mark.parametrize("n_seq", [1, 2, 5, 8])
def test_batch_matches_independent_oracle_runs(tiny_model, n_seq):
    cfg, model = tiny_model
    eng, seqs, orcs, lens, worst = _run_batch(cfg, model, n_seq)
    try:
        # every sequence's K/V rows sit at its own pages, slot pos % 16, and match its oracle cache
        from quantized_decode_gb300.kvfill import raw_view
        k, v, n_pages = eng.debug_kv()
        shape = (cfg.n_layers, n_pages, cfg.n_kv_heads, 16, cfg.head_dim)
        kp = raw_view(k, int(np.prod(shape)) * 2).view(torch.int16).view(shape).cpu().numpy().view(np.uint16)
        used = set()
        for i, s in enumerate(seqs):
            n, pages, free = eng.seq_info(s)
            assert n == lens[i] + 6 and len(pages) == (n + 15) // 16
            assert not (set(pages.tolist()) & used) and 0 not in pages
            used |= set(pages.tolist())
            rows = np.stack([kp[:, pages[p // 16], :, p % 16, :] for p in range(n)], axis=1)
            ref = orcs[i].k_cache[:, :n]
            a = synth.bf16_to_f32(rows).astype(np.float64)
            b = synth.bf16_to_f32(ref).astype(np.float64)
            assert np.max(np.abs(a - b)) <= 2e-2 * np.max(np.abs(b))
        print(f"\nbatch of {n_seq} (tiny): worst relative logit error {worst:.3e}")
    finally:
        eng.close()


def test_released_pages_are_reused_and_others_unaffected(tiny_model):
    cfg, model = tiny_model
    eng, seqs, orcs, lens, _ = _run_batch(cfg, model, 3, n_steps=2)
    try:
        _, pages1, free0 = eng.seq_info(seqs[1])
        eng.release(seqs[1])
        _, _, free1 = eng.seq_info(seqs[0])
        assert free1 == free0 + len(pages1)
        s = eng.add()                        # takes the free slot, reuses pages from the list
        assert s == seqs[1]
        prompt = sm.prompt(cfg, SEED + 9, 40, stream=9)
        eng.prefill(s, prompt)
        orc, ref = _oracle_prefix(cfg, prompt, cfg.max_context)
        check_logits(eng.logits(s), ref, "new sequence after release")
        _, pages_new, _ = eng.seq_info(s)
        assert set(pages_new.tolist()) & set(pages1.tolist())
        # the sequences that stayed continue exactly as their oracles
        for i in (0, 2):
            eng.step([seqs[i]], [5])
            check_logits(eng.logits(seqs[i]), orcs[i].step(5, lens[i] + 2), f"seq {i} after the release")
    finally:
        eng.close()


WIDE = [("qwen2.5-7b", 3), ("qwen3-8b", 2)]


@pytest.mark.parametrize("name,n_seq", WIDE, ids=[w[0] for w in WIDE])
def test_batch_full_width_two_layers(name, n_seq):
    cfg = sm.CONFIGS[name].with_(n_layers=2, max_context=256)
    model = device_model(cfg, SEED)
    eng, seqs, orcs, lens, worst = _run_batch(cfg, model, n_seq, max_seqs=4, n_steps=3,
                                              lens=[17 + 11 * i for i in range(n_seq)])
    eng.close()
    print(f"\n{name} x 2 layers, batch of {n_seq}: worst relative logit error {worst:.3e}")


def test_batch_errors(tiny_model):
    from quantized_decode_gb300 import BatchEngine, LLMError, _lib as L
    cfg, model = tiny_model
    eng = BatchEngine(model, 2, n_pages=4)          # 3 usable pages of 16 tokens
    try:
        a = eng.add()
        b = eng.add()
        with pytest.raises(LLMError) as e:
            eng.add()
        assert e.value.code == L.LLM_ERR_STATE
        with pytest.raises(LLMError) as e:
            eng.step([a])                           # nothing to feed yet
        assert e.value.code == L.LLM_ERR_STATE
        with pytest.raises(LLMError) as e:
            eng.step([a, a], [1, 2])
        assert e.value.code == L.LLM_ERR_ARG
        eng.prefill(a, sm.prompt(cfg, SEED, 32))    # two pages
        eng.prefill(b, sm.prompt(cfg, SEED, 16))    # the third
        with pytest.raises(LLMError) as e:
            eng.step([a, b], [1, 2])                # both need a new page: only none left
        assert e.value.code == L.LLM_ERR_CONTEXT_FULL
        eng.release(a)
        eng.step([b], [3])                          # takes one of a's pages
        n, pages, free = eng.seq_info(b)
        assert n == 17 and len(pages) == 2 and free == 1
    finally:
        eng.close()
