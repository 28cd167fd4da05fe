"""Full-depth teacher-forced parity at the shapes the engine is measured on (GPU required).

Every layer of each model (28 for the 7B and 1.5B shapes, 36 for Qwen3-8B), full widths and
vocabularies, directly against the CPU oracle -- never through another GPU path:
  * 7B INT4 at KV 4032 (the benchmarked configuration: one 16-CTA attention cluster per KV
    head) and at KV 8192 (several clusters per KV head and the cross-cluster combine), with the
    cache pre-filled with seeded N(0,1) K/V through a shuffled page table;
  * 1.5B INT4 (tied LM head): a 512-token prompt through the batched tensor-core prefill, then
    16 decode steps;
  * Qwen3-8B INT8 (per-row scales, q/k norms, INT8 LM head): a 128-token prompt, and a
    seeded 4096-token cache, 4 decode steps each.
Acceptance per step (the workload's parity criterion): max |GPU - oracle| <= 2e-2 *
max |oracle|, and the argmax equal wherever the oracle's top-1/top-2 margin exceeds 5e-2.
The worst relative error per configuration is printed (pytest -s / -rP shows it).
"""
import numpy as np
import pytest
import torch

import oracle
from synth import model as sm

from ._gpu import fill_kv
from .test_gpu_engine import SEED, check_logits, synth_perm

pytestmark = pytest.mark.gpu


def _pair(cfg, t_max):
    """Device model and oracle model of the same seeded weights (the large bf16 tensors are
    drawn once and handed to both)."""
    from quantized_decode_gb300 import DeviceModel
    get_proj, get_norms, emb, fin, lm = sm.recipe(cfg, SEED)
    dm = DeviceModel(cfg, get_proj, get_norms, emb, fin, lm)
    om = oracle.OracleModel(cfg, SEED, t_max=t_max, embed=emb, lm_head=lm)
    return dm, om


def _forced_steps(eng, orc, tok, pos0, n, where):
    errs = []
    for i in range(n):
        got = eng.decode_step(tok)
        ref = orc.step(tok, pos0 + i)
        errs.append(check_logits(eng.logits(), ref, f"{where} step {i}"))
        assert got == int(np.argmax(eng.logits())), where
        tok = int(np.argmax(ref))
    return errs


@pytest.fixture(scope="module")
def m7b():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    cfg = sm.CONFIGS["qwen2.5-7b"]
    dm, om = _pair(cfg, t_max=8192 + 64)
    yield cfg, dm, om


@pytest.mark.parametrize("T0,n_steps", [(4032, 4), (8192, 2)])
def test_7b_all_layers_seeded_cache(m7b, T0, n_steps):
    from quantized_decode_gb300 import Engine, make_config
    cfg0, dm, orc = m7b
    cfg = cfg0.with_(max_context=max(cfg0.max_context, T0 + 64))
    eng = Engine(dm, config=make_config(cfg))       # the weights are the 7B model's either way
    try:
        ks, vs = fill_kv(eng, cfg, 31, T0, page_perm=synth_perm((cfg.max_context + 15) // 16))
        for l in range(cfg.n_layers):
            orc.set_kv(l, ks[l], vs[l])
        errs = _forced_steps(eng, orc, 7, T0, n_steps, f"7B KV {T0}")
        print(f"\n7B x {cfg.n_layers} layers, KV {T0}: worst relative logit error {max(errs):.3e}")
    finally:
        eng.close()


def test_1p5b_all_layers_pp512_then_16_steps():
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS["qwen2.5-1.5b"].with_(max_context=1024)
    dm, orc = _pair(cfg, t_max=1024)
    eng = Engine(dm)
    try:
        prompt = sm.prompt(cfg, SEED, 512)
        first = eng.prefill(prompt)                      # batched tensor-core prefill
        ref = orc.prefill(prompt)
        errs = [check_logits(eng.logits(), ref, "1.5B pp512 prefill")]
        assert first == int(np.argmax(eng.logits()))
        errs += _forced_steps(eng, orc, int(np.argmax(ref)), 512, 16, "1.5B")
        print(f"\n1.5B x {cfg.n_layers} layers, pp512 + 16: worst relative logit error {max(errs):.3e}")
    finally:
        eng.close()


@pytest.fixture(scope="module")
def q3():
    cfg = sm.CONFIGS["qwen3-8b"]
    dm, om = _pair(cfg, t_max=cfg.max_context)
    yield cfg, dm, om


def test_qwen3_8b_all_layers_input_128(q3):
    from quantized_decode_gb300 import Engine
    cfg, dm, orc = q3
    eng = Engine(dm)
    try:
        prompt = sm.prompt(cfg, SEED, 128)
        first = eng.prefill(prompt)
        ref = orc.prefill(prompt)
        errs = [check_logits(eng.logits(), ref, "Qwen3-8B input 128 prefill")]
        assert first == int(np.argmax(eng.logits()))
        errs += _forced_steps(eng, orc, int(np.argmax(ref)), 128, 4, "Qwen3-8B input 128")
        print(f"\nQwen3-8B x {cfg.n_layers} layers, input 128 + 4: worst relative logit error {max(errs):.3e}")
    finally:
        eng.close()


def test_qwen3_8b_all_layers_seeded_cache_4096(q3):
    from quantized_decode_gb300 import Engine
    cfg, dm, orc = q3
    eng = Engine(dm)
    try:
        T0 = 4096
        ks, vs = fill_kv(eng, cfg, 37, T0, page_perm=synth_perm((cfg.max_context + 15) // 16))
        for l in range(cfg.n_layers):
            orc.set_kv(l, ks[l], vs[l])
        errs = _forced_steps(eng, orc, 11, T0, 4, "Qwen3-8B KV 4096")
        print(f"\nQwen3-8B x {cfg.n_layers} layers, KV 4096: worst relative logit error {max(errs):.3e}")
    finally:
        eng.close()
