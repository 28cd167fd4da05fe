"""The MLP block as one kernel (llm_set_fused_mlp) against the oracle and against the two
GEMV kernels (GPU required).

The fused kernel adds the CTAs' down-projection partial sums in 64-bit fixed point, so its
results must repeat bit for bit; against the oracle it must meet the acceptance rule
(max |GPU - oracle| <= 2e-2 max |oracle|, argmax equal where the top-1/top-2 margin > 5e-2),
and against the two-kernel path it differs only by rounding (1e-3 of the logit scale).
Shapes: the tiny model (INT4), the 7B width (INT4, 2 layers, full vocabulary, seeded cache
through a shuffled page table) and the Qwen3-8B width (INT8 with per-row scales, q/k norms).
"""
import numpy as np
import pytest
import torch

import oracle
from synth import model as sm

from ._gpu import device_model, fill_kv
from .test_gpu_engine import SEED, check_logits, synth_perm

pytestmark = pytest.mark.gpu

CASES = [("tiny", 2, 200), ("qwen2.5-7b", 2, 1000), ("qwen3-8b", 2, 700)]


@pytest.mark.parametrize("name,n_layers,T0", CASES, ids=[c[0] for c in CASES])
def test_fused_mlp_vs_oracle_and_two_kernels(name, n_layers, T0):
    from quantized_decode_gb300 import Engine
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    cfg = sm.CONFIGS[name].with_(n_layers=n_layers)
    eng = Engine(device_model(cfg, SEED))
    try:
        ks, vs = fill_kv(eng, cfg, 41, T0, page_perm=synth_perm((cfg.max_context + 15) // 16))
        runs = {}
        for fused in (True, False, True):
            eng.set_fused_mlp(fused)
            eng.debug_kv(set_len=T0)
            orc = oracle.OracleModel(cfg, SEED, t_max=T0 + 8)
            for l in range(cfg.n_layers):
                orc.set_kv(l, ks[l], vs[l])
            tok, out = 5, []
            for i in range(4):
                got = eng.decode_step(tok)
                ref = orc.step(tok, T0 + i)
                check_logits(eng.logits(), ref, f"{name} fused={fused} step {i}")
                assert got == int(np.argmax(eng.logits()))
                out.append(eng.logits().copy())
                tok = int(np.argmax(ref))
            if fused in runs:   # the second fused run repeats the first bit for bit
                for a, b in zip(runs[fused], out):
                    np.testing.assert_array_equal(a, b)
            runs[fused] = out
        for a, b in zip(runs[True], runs[False]):
            assert float(np.max(np.abs(a - b))) <= 1e-3 * float(np.max(np.abs(b)))
    finally:
        eng.close()


def test_fused_mlp_refuses_shapes_it_does_not_take():
    from quantized_decode_gb300 import Engine, LLMError, _lib as L
    cfg = sm.CONFIGS["tiny"].with_(hidden=4608, n_q_heads=36, n_kv_heads=6, head_dim=128,
                                   mlp=768, n_layers=1, vocab=1024)   # hidden 4608 > 4096
    eng = Engine(device_model(cfg, SEED))
    try:
        with pytest.raises(LLMError) as e:
            eng.set_fused_mlp(True)
        assert e.value.code == L.LLM_ERR_ARG
        eng.set_fused_mlp(False)
    finally:
        eng.close()


def test_step_kinds_follow_the_mode():
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS["tiny"]
    eng = Engine(device_model(cfg, SEED))
    try:
        eng.set_fused_mlp(True)
        assert eng.step_kinds() == ["qkv", "attention", "o_proj", "mlp"] * cfg.n_layers + ["lm_head"]
        eng.set_fused_mlp(False)
        assert eng.step_kinds() == ["qkv", "attention", "o_proj", "gate_up", "down"] * cfg.n_layers + ["lm_head"]
    finally:
        eng.close()
