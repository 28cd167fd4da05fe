"""An engine created from a model file against one created from the same weights in device
memory (GPU required): identical tokens and bit-identical logits, the context override, and
no leak across create/destroy."""
import numpy as np
import pytest
import torch

from synth import model as sm

from ._gpu import device_model
from .test_gpu_engine import SEED
from .test_model_file import TINY8

pytestmark = pytest.mark.gpu


def _run(eng, prompt, n):
    eng.reset()
    toks = [eng.prefill(prompt)]
    logits = [eng.logits()]
    for _ in range(n):
        toks.append(eng.decode_step())
        logits.append(eng.logits())
    return toks, np.stack(logits)


@pytest.mark.parametrize("cfg", [sm.CONFIGS["tiny"], TINY8], ids=["tiny-int4", "tiny-int8"])
def test_file_engine_equals_device_engine(tmp_path, cfg):
    from quantized_decode_gb300 import Engine, write_model_file
    assert torch.cuda.is_available()
    path = tmp_path / "m.qd"
    write_model_file(path, cfg, *sm.recipe(cfg, SEED))
    prompt = sm.prompt(cfg, SEED, 20)
    a = Engine(device_model(cfg, SEED))
    ta, la = _run(a, prompt, 12)
    a.close()
    b = Engine.from_file(path)
    tb, lb = _run(b, prompt, 12)
    b.close()
    assert ta == tb
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))


def test_file_engine_context_override_and_cleanup(tmp_path):
    from quantized_decode_gb300 import Engine, LLMError, write_model_file, _lib as L
    cfg = sm.CONFIGS["tiny"]
    path = tmp_path / "m.qd"
    write_model_file(path, cfg, *sm.recipe(cfg, SEED))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        e = Engine.from_file(path, max_context=24)
        assert e.cfg.max_context == 24
        e.prefill(sm.prompt(cfg, SEED, 20))
        for _ in range(4):
            e.decode_step()
        with pytest.raises(LLMError) as err:
            e.decode_step()
        assert err.value.code == L.LLM_ERR_CONTEXT_FULL
        e.close()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - (8 << 20)
