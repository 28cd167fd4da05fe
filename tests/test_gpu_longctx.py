"""Long-context decode through the C ABI against the CPU oracle (GPU required).

The workload's long-context stress: the 7B shape (two layers here, full widths and vocabulary)
with the paged bf16 KV cache pre-filled to 8192, 16384 and 32768 tokens of seeded N(0,1) K/V
through a shuffled, non-contiguous page table, then teacher-forced greedy steps; the split-K
attention derives each split's pages from the current length.  Acceptance as in the engine tests:
max |GPU - oracle| <= 2e-2 * max |oracle|, argmax equal where the top-1/top-2 margin > 5e-2.
"""
import numpy as np
import pytest

import oracle
from synth import model as sm

from ._gpu import device_model, fill_kv
from .test_gpu_engine import SEED, check_logits, synth_perm

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T0", [8192, 16384, 32768])
def test_long_context_two_layers_vs_oracle(T0):
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS["qwen2.5-7b"].with_(n_layers=2, max_context=32768 + 64)
    eng = Engine(device_model(cfg, SEED))
    try:
        n_pages = (cfg.max_context + 15) // 16
        ks, vs = fill_kv(eng, cfg, 17, T0, page_perm=synth_perm(n_pages))
        orc = oracle.OracleModel(cfg, SEED, t_max=T0 + 4)
        for l in range(cfg.n_layers):
            orc.set_kv(l, ks[l], vs[l])
        tok = 11
        for i in range(2):
            got = eng.decode_step(tok)
            ref = orc.step(tok, T0 + i)
            check_logits(eng.logits(), ref, f"T0={T0} step {i}")
            assert got == int(np.argmax(eng.logits()))
            tok = int(np.argmax(ref))
    finally:
        eng.close()
