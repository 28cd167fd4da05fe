"""INT4 GEMVs on int8 activations (GPU required): the op against the oracle's definition, and
the decode step with llm_set_act_int8 against the FP32 oracle within the acceptance tolerance.

The activation codes are decided in fp32 on both sides (same quotient, same rounding), so the op
differs from the oracle only by the fp32 accumulation of exact integer dots times the scales:
|err| <= 2e-5 * sum_g |s_w sx| sum_k |c q| (the per-unit sums are accumulated in fp32, a few
hundred terms at most, each rounded once)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import act_int8 as oa
from synth import model as sm

from ._gpu import device_model, to_dev
from .test_gpu_engine import LOGIT_TOL, SEED, _teacher_forced

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import quantized_decode_gb300 as qd
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return qd.load()


def _op(lib, codes, scales, x):
    import quantized_decode_gb300 as qd
    N, K = codes.shape
    w, s = to_dev(qd.pack_int4(codes)), to_dev(scales)
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    assert lib.llm_op_gemv_int4_a8(w.data_ptr(), s.data_ptr(), N, K, xd.data_ptr(), y.data_ptr(), None) == 0
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("N,K", [(32, 256), (256, 1024), (3584, 3584), (3584, 18944), (1536, 8960),
                                 (4608, 3584)])
def test_op_matches_the_oracle(lib, N, K):
    codes, scales = sm.quantized_tensor(sm.FMT_INT4_G128, 31, N + K, N, K)
    x = synth.normal_f32(32, K, K, 0.0, 1.0)
    x[128:256] = 0.0                                     # a zero group
    x[256:384] *= 1e3
    if K > 512:
        x[512:640] *= 1e-6
    y = _op(lib, codes, scales, x)
    ref, mag = oa.gemv_int4_a8(codes, scales, x)
    err = np.abs(y - ref)
    assert np.all(err <= 2e-5 * mag + 1e-30), float(np.max(err / (mag + 1e-30)))


def test_op_rejects_bad_shapes(lib):
    from quantized_decode_gb300 import _lib as L
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    for N, K in ((32, 128), (30, 256), (32, 65536)):
        assert lib.llm_op_gemv_int4_a8(p, p, N, K, p, p, None) == L.LLM_ERR_ARG


@pytest.mark.parametrize("name", ["tiny", "qwen2.5-7b"])
def test_decode_with_int8_activations_vs_fp32_oracle(name):
    from quantized_decode_gb300 import Engine
    cfg = sm.CONFIGS[name] if name == "tiny" else sm.CONFIGS[name].with_(n_layers=2)
    eng = Engine(device_model(cfg, SEED))
    eng.set_act_int8(True)
    orc = oracle.OracleModel(cfg, SEED)
    errs = _teacher_forced(cfg, eng, orc, 24 if name == "tiny" else 8, 12 if name == "tiny" else 4)
    assert max(errs) < LOGIT_TOL
    # the variant changes the logits (the activations are rounded), and switching back restores them
    eng.set_act_int8(False)
    errs0 = _teacher_forced(cfg, eng, orc, 8, 2)
    assert max(errs0) < LOGIT_TOL
    eng.close()


def test_switch_refusals():
    from quantized_decode_gb300 import Engine, LLMError, _lib as L
    cfg = sm.CONFIGS["qwen3-8b"].with_(n_layers=1, hidden=512, n_q_heads=4, n_kv_heads=2, mlp=1024,
                                        vocab=1024, max_context=64)
    eng = Engine(device_model(cfg, SEED))                # INT8 weights: no int8-activation variant
    with pytest.raises(LLMError) as e:
        eng.set_act_int8(True)
    assert e.value.code == L.LLM_ERR_ARG
    eng.set_act_int8(False)
    eng.close()
