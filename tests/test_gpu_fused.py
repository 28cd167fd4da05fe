"""The fused QKV projection + attention kernel (one 16-CTA cluster per KV head) against the
CPU oracle and against the separate QKV and attention kernels (GPU required).

Shapes: the 7B (G = 7, K = 3584: 8 warps split K) and 1.5B (G = 6, K = 1536: tile slots of
2 warps) widths with 2 layers; positions from 0 (one page, 15 CTAs of each cluster without
pages) across page boundaries, and a seeded cache of 1000 tokens through a shuffled table.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import model as sm

from ._gpu import device_model, fill_kv, kv_pool_views
from .test_gpu_engine import SEED, check_logits

pytestmark = pytest.mark.gpu

SHAPES = ["qwen2.5-7b", "qwen2.5-1.5b"]


@pytest.fixture(scope="module", params=SHAPES)
def shape(request):
    from quantized_decode_gb300 import Engine
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    cfg = sm.CONFIGS[request.param].with_(n_layers=2)
    eng = Engine(device_model(cfg, SEED))
    eng.set_fused_attention(True)           # raises if the model does not take the fused kernel
    yield cfg, eng
    eng.close()


def _identity_table(eng, cfg):
    kp, vp, ptv = kv_pool_views(eng, cfg)
    ptv.copy_(torch.arange(ptv.numel(), dtype=torch.int32, device="cuda"))


def test_from_position_zero_vs_oracle(shape):
    """Teacher-forced steps from an empty cache: T = 1 leaves 15 CTAs of every cluster
    without a page; 20 steps cross the first page boundary."""
    cfg, eng = shape
    _identity_table(eng, cfg)
    eng.reset()
    orc = oracle.OracleModel(cfg, SEED, t_max=24)
    tok = 11
    for pos in range(20):
        eng.decode_step(tok)
        ref = orc.step(tok, pos)
        check_logits(eng.logits(), ref, f"pos {pos}")
        tok = int(np.argmax(ref))
    # the K/V rows the fused kernel appended equal the oracle's cache (bf16)
    kp, vp, ptv = kv_pool_views(eng, cfg)
    table = ptv.cpu().numpy()
    for pool, ref in ((kp, orc.k_cache), (vp, orc.v_cache)):
        arr = pool.cpu().numpy().view(np.uint16)
        got = np.stack([arr[:, table[p // 16], :, p % 16, :] for p in range(20)], axis=1)
        g = (got.astype(np.uint32) << 16).view(np.float32)
        r = (ref[:, :20].astype(np.uint32) << 16).view(np.float32)
        assert np.max(np.abs(g - r)) <= 2e-2 * np.max(np.abs(r))
    eng.reset()


def test_seeded_cache_through_shuffled_pages_vs_oracle(shape):
    cfg, eng = shape
    T0 = 1000
    eng.reset()
    n_pages = (cfg.max_context + 15) // 16
    ks, vs = fill_kv(eng, cfg, 9, T0, page_perm=synth.permutation(SEED, 4, n_pages))
    orc = oracle.OracleModel(cfg, SEED, t_max=T0 + 8)
    for l in range(cfg.n_layers):
        orc.set_kv(l, ks[l], vs[l])
    tok = 5
    for i in range(6):
        eng.decode_step(tok)
        ref = orc.step(tok, T0 + i)
        check_logits(eng.logits(), ref, f"step {i}")
        tok = int(np.argmax(ref))
    _identity_table(eng, cfg)
    eng.reset()


def test_fused_equals_separate_kernels(shape):
    """Same cache and tokens through both paths.  The projection's K parts are summed in
    another order (fp32, ~1e-6 relative), which can flip the bf16 rounding of an appended
    K/V element by one ulp (2^-8 relative); over a few steps that moves the logits by
    ~1e-3 of their scale, so the bound is a quarter of the oracle acceptance (5e-3)."""
    cfg, eng = shape
    T0 = 333
    out = {}
    for fused in (True, False):
        eng.set_fused_attention(fused)
        eng.reset()
        fill_kv(eng, cfg, 13, T0)
        toks, logits = [], []
        tok = 7
        for i in range(5):
            tok = eng.decode_step(tok)
            toks.append(tok)
            logits.append(eng.logits())
        out[fused] = (toks, np.stack(logits))
    eng.set_fused_attention(True)
    (t1, l1), (t0, l0) = out[True], out[False]
    scale = float(np.max(np.abs(l0)))
    assert float(np.max(np.abs(l1 - l0))) <= 5e-3 * scale
    for a, b, lg in zip(t1, t0, l0):
        top2 = np.sort(lg)[-2:]
        if top2[1] - top2[0] > 5e-2:
            assert a == b
    eng.reset()


def test_models_outside_the_fused_kernel_are_refused():
    """head_dim 64 (the tiny shape) does not take the fused kernel."""
    from quantized_decode_gb300 import Engine, LLMError, _lib as L
    cfg = sm.CONFIGS["tiny"]
    eng = Engine(device_model(cfg, SEED))
    try:
        with pytest.raises(LLMError) as e:
            eng.set_fused_attention(True)
        assert e.value.code == L.LLM_ERR_ARG
        eng.set_fused_attention(False)
    finally:
        eng.close()
