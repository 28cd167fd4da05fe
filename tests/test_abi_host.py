"""Host-side checks of the C ABI that need no GPU: exported symbols, the offline packer
against the oracle's packer (bit-exact), and argument validation that returns before any
CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth
from synth import model as sm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import quantized_decode_gb300 as qd
    qd.build()
    return qd.load()


def _declared_functions():
    names = []
    for hdr in ("llm.h", "llm_ops.h"):
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?(?:int|void|char)\s*\*?\s*(llm_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 19, names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_every_declared_symbol():
    from quantized_decode_gb300 import _lib
    assert set(_declared_functions()) == set(_lib.SIGNATURES)


@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (64, 3584), (3, 18944)])
def test_packer_matches_oracle_bit_exact(lib, N, K):
    import quantized_decode_gb300 as qd
    codes = synth.randint_i8(N, K, N * K, -8, 7).reshape(N, K)
    assert np.array_equal(qd.pack_int4(codes), oracle.pack_int4(codes))


def test_packer_golden_and_range_check(lib):
    import quantized_decode_gb300 as qd
    codes = np.zeros((1, 128), np.int8)
    codes[0, :8] = np.arange(8)
    assert int(qd.pack_int4(codes)[0, 0]) == 0x75316420
    codes[0, 5] = 8
    with pytest.raises(qd.LLMError):
        qd.pack_int4(codes)
    bad = np.full((2, 128), -128, np.int8)
    with pytest.raises(qd.LLMError):
        qd.pack_int8(bad)
    ok = synth.randint_i8(1, 2, 2 * 128, -127, 127).reshape(2, 128)
    assert np.array_equal(qd.pack_int8(ok), ok)


def _tiny_struct(**over):
    from quantized_decode_gb300 import make_config
    c = make_config(sm.CONFIGS["tiny"])
    for k, v in over.items():
        setattr(c, k, v)
    return c


def _fake_weights(n_layers, addr=0x10000):
    from quantized_decode_gb300 import _lib
    layers = (_lib.llm_layer_weights * n_layers)()
    for l in range(n_layers):
        for i, f in enumerate(_lib.LAYER_FIELDS):
            setattr(layers[l], f, addr + 4096 * (l * 32 + i))
    w = _lib.llm_weights(addr, addr + 256, addr + 512, 0, layers)
    return w, layers


def _create(lib, cfg, w):
    h = ctypes.c_void_p()
    return lib.llm_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(h)), h


def test_create_refuses_layout_mismatch_before_touching_the_gpu(lib):
    from quantized_decode_gb300 import _lib as L
    w, keep = _fake_weights(2)
    rc, h = _create(lib, _tiny_struct(layout_id=L.LLM_LAYOUT_INT8_ROW), w)
    assert rc == L.LLM_ERR_LAYOUT and not h.value
    rc, _ = _create(lib, _tiny_struct(weight_format=2, layout_id=1), w)
    assert rc == L.LLM_ERR_LAYOUT


@pytest.mark.parametrize("field,value", [("page_tokens", 32), ("head_dim", 96), ("n_kv_heads", 3),
                                         ("hidden", 200), ("max_context", 0), ("vocab", 1000),
                                         ("weight_format", 9), ("rope_base", 0.0)])
def test_create_rejects_bad_config(lib, field, value):
    from quantized_decode_gb300 import _lib as L
    w, keep = _fake_weights(2)
    rc, h = _create(lib, _tiny_struct(**{field: value}), w)
    assert rc == L.LLM_ERR_ARG and not h.value


def test_create_rejects_null_and_misaligned_pointers(lib):
    from quantized_decode_gb300 import _lib as L
    w, layers = _fake_weights(2)
    layers[1].wd = 0x10008          # not 16-byte aligned
    assert _create(lib, _tiny_struct(), w)[0] == L.LLM_ERR_ARG
    w, layers = _fake_weights(2)
    layers[0].bq = None             # bias required by the config
    assert _create(lib, _tiny_struct(), w)[0] == L.LLM_ERR_ARG
    h = ctypes.c_void_p()
    assert lib.llm_create(None, None, None, ctypes.byref(h)) == L.LLM_ERR_ARG


def test_null_handles_and_status_strings(lib):
    from quantized_decode_gb300 import _lib as L
    lib.llm_destroy(None)
    out = ctypes.c_int32()
    assert lib.llm_decode_step(None, -1, ctypes.byref(out)) == L.LLM_ERR_ARG
    assert lib.llm_reset(None) == L.LLM_ERR_ARG
    for code in range(0, -10, -1):
        assert lib.llm_status_str(code) != b"unknown status", code
    assert b"context" in lib.llm_status_str(L.LLM_ERR_CONTEXT_FULL)
    assert b"model file" in lib.llm_status_str(L.LLM_ERR_FORMAT)
    assert lib.llm_set_sampling(None, 0.6, 20, 0.95, 1) == L.LLM_ERR_ARG
    assert lib.llm_set_act_int8(None, 1) == L.LLM_ERR_ARG


def test_new_ops_refuse_bad_arguments_before_any_launch(lib):
    """Argument checks that return before any CUDA call (no GPU here)."""
    from quantized_decode_gb300 import _lib as L
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16   # 16-byte aligned host address
    tok = ctypes.c_int32()
    for V, T, k, top_p in ((0, 1.0, 1, 1.0), (100, 0.0, 5, 0.9), (100, float("inf"), 5, 0.9), (100, 1.0, 0, 0.9),
                           (100, 1.0, 101, 0.9), (2000, 1.0, 1025, 0.9), (100, 1.0, 5, 0.0), (100, 1.0, 5, 1.5)):
        assert lib.llm_op_sample(p, V, T, k, top_p, 1, 0, ctypes.byref(tok), None) == L.LLM_ERR_ARG
    assert lib.llm_op_sample(None, 100, 1.0, 5, 0.9, 1, 0, ctypes.byref(tok), None) == L.LLM_ERR_ARG
    for N, K in ((32, 128), (30, 256), (32, 65536), (0, 256)):
        assert lib.llm_op_gemv_int4_a8(p, p, N, K, p, p, None) == L.LLM_ERR_ARG
    assert lib.llm_op_gemv_int4_a8(p + 4, p, 32, 256, p, p, None) == L.LLM_ERR_ARG   # misaligned codes
    assert lib.llm_op_gemv_int4_a8(p, None, 32, 256, p, p, None) == L.LLM_ERR_ARG


def test_synthetic_scales_give_rms_002():
    cfg = sm.CONFIGS["tiny"]
    t = sm.layer_proj(cfg, 3, 0, "gate")
    W = t["codes"].astype(np.float64) * np.repeat(synth.bf16_to_f32(t["scales"]), 128, axis=1)
    assert abs(np.sqrt(np.mean(W ** 2)) - 0.02) < 0.0005
    codes, scales = sm.quantized_tensor(sm.FMT_INT8_ROW, 3, 9, 256, 512)
    W8 = codes.astype(np.float64) * scales[:, None]
    assert abs(np.sqrt(np.mean(W8 ** 2)) - 0.02) < 0.0005
