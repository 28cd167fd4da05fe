"""o_proj folded into the decode attention clusters (llm_set_o_fold), GPU required.

The folded step must meet the acceptance rule against the oracle on its own (every step, full
widths of the 7B shape, a seeded cache through a shuffled page table), stay close to the
unfolded chain, give bitwise the same logits when a step is repeated (the fixed-point row sums
do not depend on the order of the CTAs), and be refused where the attention plan or the weight
format does not allow it.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import model as sm

from ._gpu import device_model, fill_kv
from .test_gpu_engine import SEED, check_logits, synth_perm

pytestmark = pytest.mark.gpu


def _pair(cfg, t_max):
    from quantized_decode_gb300 import DeviceModel
    get_proj, get_norms, emb, fin, lm = sm.recipe(cfg, SEED)
    dm = DeviceModel(cfg, get_proj, get_norms, emb, fin, lm)
    om = oracle.OracleModel(cfg, SEED, t_max=t_max, embed=emb, lm_head=lm)
    return dm, om


@pytest.mark.parametrize("layers,T0", [(2, 300), (4, 2049)])
def test_folded_step_vs_oracle_7b_widths(layers, T0):
    from quantized_decode_gb300 import Engine
    assert torch.cuda.is_available()
    cfg = sm.CONFIGS["qwen2.5-7b"].with_(n_layers=layers)
    dm, orc = _pair(cfg, t_max=T0 + 16)
    eng = Engine(dm)
    try:
        eng.set_o_fold(True)
        ks, vs = fill_kv(eng, cfg, 31, T0, page_perm=synth_perm((cfg.max_context + 15) // 16))
        for l in range(cfg.n_layers):
            orc.set_kv(l, ks[l], vs[l])
        tok = 11
        for i in range(4):
            got = eng.decode_step(tok)
            ref = orc.step(tok, T0 + i)
            check_logits(eng.logits(), ref, f"folded o_proj, {layers} layers, step {i}")
            assert got == int(np.argmax(eng.logits()))
            tok = int(np.argmax(ref))
        # the same step again, folded and unfolded
        eng.truncate(T0 + 3)
        eng.decode_step(tok)
        a = eng.logits()
        eng.truncate(T0 + 3)
        eng.decode_step(tok)
        assert np.array_equal(a, eng.logits()), "the folded step is not repeatable bit for bit"
        eng.set_o_fold(False)
        eng.truncate(T0 + 3)
        eng.decode_step(tok)
        b = eng.logits()
        assert float(np.max(np.abs(a - b))) <= 2e-2 * float(np.max(np.abs(b)))
    finally:
        eng.close()


def test_fold_refused_where_it_does_not_apply():
    from quantized_decode_gb300 import Engine, LLMError
    eng = Engine(device_model(sm.CONFIGS["tiny"], SEED))        # head_dim 64
    try:
        with pytest.raises(LLMError):
            eng.set_o_fold(True)
        eng.set_o_fold(False)
    finally:
        eng.close()
