"""Temperature / top-k / top-p sampling on the GPU against the oracle's sampler (GPU required).

The GPU computes the weights and running sums in float32, the oracle in float64, so a draw can
differ only when it falls within rounding of a boundary: tokens are compared wherever the
oracle's relative decision margin exceeds 1e-4 (far above float32 rounding of sums of at most
1024 weights in [0, 1]), and every GPU token must lie in the oracle's kept (top-k, top-p) set.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import sampling as smp
from synth import model as sm

from ._gpu import device_model, to_dev
from .test_gpu_engine import SEED

pytestmark = pytest.mark.gpu

MARGIN = 1e-4


@pytest.fixture(scope="module")
def lib():
    import quantized_decode_gb300 as qd
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return qd.load()


def _op(lib, logits_dev, V, T, k, p, seed, counter):
    tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    assert lib.llm_op_sample(logits_dev.data_ptr(), V, T, k, p, seed, counter, tok.data_ptr(), None) == 0
    torch.cuda.synchronize()
    return int(tok.item())


@pytest.mark.parametrize("V", [152064, 1000])
@pytest.mark.parametrize("T,k,p", [(0.6, 20, 0.95), (1.0, 1, 1.0), (1.5, 1000, 0.9), (0.3, 50, 1.0),
                                   (1.0, 7, 0.5), (2.0, 256, 0.99)])
def test_op_matches_oracle(lib, V, T, k, p):
    logits = synth.normal_f32(V + k, 7, V, 0.0, 3.0)
    dev = to_dev(logits)
    compared = 0
    for counter in range(40):
        got = _op(lib, dev, V, T, k, p, 321, counter)
        tok, kept, margin = smp.sample(logits, T, k, p, 321, counter)
        assert got in kept, (counter, got)
        if margin > MARGIN:
            assert got == tok, (counter, got, tok, margin)
            compared += 1
    assert compared >= 30


def _compare(lib, logits, dev_ptr, V, T, k, p, seed, n_draws, min_compared):
    compared = 0
    for counter in range(n_draws):
        tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        assert lib.llm_op_sample(dev_ptr, V, T, k, p, seed, counter, tok.data_ptr(), None) == 0
        torch.cuda.synchronize()
        got = int(tok.item())
        want, kept, margin = smp.sample(logits, T, k, p, seed, counter)
        assert got in kept, (counter, got)
        if margin > MARGIN:
            assert got == want, (counter, got, want, margin)
            compared += 1
    assert compared >= min_compared


def test_op_one_dense_bin_takes_the_sorting_path(lib):
    """3000 logits within one 12-bit key bin ([1, 1.0625)): every key is a candidate of the same
    bin, so the candidates are sorted instead of ranked within their bin."""
    V = 3000
    u = synth.normal_f32(V, 11, V, 0.0, 1.0)
    logits = (1.0 + 0.06 * (0.5 + 0.5 * np.tanh(u))).astype(np.float32)
    assert logits.min() >= 1.0 and logits.max() < 1.0625
    dev = to_dev(logits)
    for T, k, p in ((0.05, 100, 0.9), (0.01, 1000, 1.0), (1.0, 7, 0.5)):
        _compare(lib, logits, dev.data_ptr(), V, T, k, p, 9, 30, 20)


def test_op_unaligned_logits_take_the_word_path(lib):
    """Logits that do not start on a 16-byte boundary are read a word at a time."""
    V = 40001
    logits = synth.normal_f32(V + 1, 13, V + 1, 0.0, 2.0)
    dev = to_dev(logits)
    for T, k, p in ((0.6, 20, 0.95), (1.5, 1000, 0.9)):
        _compare(lib, logits[1:], dev.data_ptr() + 4, V, T, k, p, 4, 30, 20)


def test_op_ties_at_the_threshold_keep_the_lowest_indices(lib):
    V = 5000
    logits = np.zeros(V, np.float32)
    logits[[17, 4000]] = 1.0                 # two above, the rest tied below
    dev = to_dev(logits)
    seen = set()
    for counter in range(200):
        t = _op(lib, dev, V, 1.0, 10, 1.0, 5, counter)
        seen.add(t)
        _, kept, _ = smp.sample(logits, 1.0, 10, 1.0, 5, counter)
        assert t in kept
    assert seen <= {17, 4000, 0, 1, 2, 3, 4, 5, 6, 7}


def test_op_rejects_bad_arguments(lib):
    from quantized_decode_gb300 import _lib as L
    dev = to_dev(np.zeros(100, np.float32))
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T, k, p in ((0.0, 5, 0.9), (1.0, 0, 0.9), (1.0, 101, 0.9), (1.0, 1025, 0.9), (1.0, 5, 0.0),
                    (1.0, 5, 1.5)):
        assert lib.llm_op_sample(dev.data_ptr(), 100, T, k, p, 1, 0, tok.data_ptr(), None) == L.LLM_ERR_ARG


@pytest.fixture(scope="module")
def tiny():
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS["tiny"]
    eng = Engine(device_model(cfg, SEED))
    yield cfg, eng
    eng.set_sampling(0.0)
    eng.close()


def _run(eng, cfg, prompt, n, forced=None):
    eng.reset()
    toks = [eng.prefill(prompt)]
    logits = [eng.logits()]
    for i in range(n):
        toks.append(eng.decode_step() if forced is None else eng.decode_step(forced[i]))
        logits.append(eng.logits())
    return toks, logits


def test_engine_draws_match_the_oracle_on_its_own_logits(tiny):
    """Each step's token is the oracle's draw from that step's logits with the draw number =
    the position whose logits are sampled (the prompt's last position for the first token)."""
    cfg, eng = tiny
    T, k, p, seed = 0.8, 40, 0.9, 1234
    eng.set_sampling(T, k, p, seed)
    prompt = sm.prompt(cfg, SEED, 12)
    toks, logits = _run(eng, cfg, prompt, 30)
    compared = 0
    for i, (t, lg) in enumerate(zip(toks, logits)):
        pos = len(prompt) - 1 + i
        tok, kept, margin = smp.sample(lg, T, k, p, seed, pos)
        assert t in kept, i
        if margin > MARGIN:
            assert t == tok, (i, t, tok, margin)
            compared += 1
    assert compared >= 25
    eng.set_sampling(0.0)


def test_engine_sampling_is_reproducible_and_seeded(tiny):
    cfg, eng = tiny
    prompt = sm.prompt(cfg, SEED, 9)
    eng.set_sampling(1.0, 50, 0.95, 77)
    a = _run(eng, cfg, prompt, 20)[0]
    b = _run(eng, cfg, prompt, 20)[0]
    eng.set_sampling(1.0, 50, 0.95, 78)
    c = _run(eng, cfg, prompt, 20)[0]
    eng.set_sampling(0.0)
    greedy = _run(eng, cfg, prompt, 20)[0]
    assert a == b
    assert a != c
    assert a != greedy


def test_engine_sampling_arguments(tiny):
    from quantized_decode_gb300 import LLMError, _lib as L
    cfg, eng = tiny
    for args in ((1.0, 0, 0.9, 1), (1.0, cfg.vocab + 1, 0.9, 1), (1.0, 5, 1.5, 1), (1.0, 5, 0.0, 1)):
        with pytest.raises(LLMError) as e:
            eng.set_sampling(*args)
        assert e.value.code == L.LLM_ERR_ARG
    eng.set_sampling(0.0)
