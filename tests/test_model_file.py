"""Offline quantizers and the model file, on the CPU.

The oracle's quantizers are pinned by hand examples (exact scales, ties, zero groups, the bf16
rounding of a scale); the library's quantizers must match them bit for bit.  The model file is
checked against its documented map: size, header fields, every tensor at its 128-byte-aligned
offset, zero padding, and the refusals (magic, version, checksum, layout id, truncation)."""
import ctypes
import os

import numpy as np
import pytest

from oracle import quantize as oq
from synth import model as sm


@pytest.fixture(scope="module")
def qd():
    import quantized_decode_gb300 as qd
    qd.build()
    return qd


# ---- oracle pins -----------------------------------------------------------------------------

def test_oracle_int4_exact_multiples_of_a_bf16_scale():
    codes = np.tile(np.arange(-7, 8), 9)[:128].astype(np.float32)
    w = (codes * 0.5).reshape(1, 128)                       # absmax 3.5 -> scale 0.5 exactly
    q, s = oq.quantize_int4_g128(w)
    assert oq.bf16_bits_to_f32(s)[0, 0] == 0.5
    assert np.array_equal(q[0], codes.astype(np.int8))


def test_oracle_int4_rounds_half_to_even_and_never_emits_minus_8():
    w = np.zeros((1, 128), np.float32)
    w[0, :6] = [7.0, 2.5, 3.5, -0.5, 1.5, -7.0]             # scale 1
    q, s = oq.quantize_int4_g128(w)
    assert oq.bf16_bits_to_f32(s)[0, 0] == 1.0
    assert list(q[0, :6]) == [7, 2, 4, 0, 2, -7]
    assert q.min() >= -7


def test_oracle_int4_scale_is_the_bf16_rounding_of_absmax_over_7():
    w = np.zeros((1, 256), np.float32)
    w[0, 0], w[0, 1] = 1.0, -1.0                            # group 0: absmax 1; group 1: zeros
    q, s = oq.quantize_int4_g128(w)
    # 1/7 = 0x3E124925 in fp32; the dropped half 0x4925 < 0x8000 -> bf16 0x3E12
    assert s[0, 0] == 0x3E12 and s[0, 1] == 0
    assert q[0, 0] == 7 and q[0, 1] == -7                   # 1 / 0.142578125 = 7.01
    assert not q[0, 128:].any()


def test_oracle_int4_error_is_at_most_half_a_step():
    rng = np.random.default_rng(3)
    w = rng.normal(0, 0.02, (64, 512)).astype(np.float32)
    q, s = oq.quantize_int4_g128(w)
    sc = np.repeat(oq.bf16_bits_to_f32(s), 128, axis=1)
    assert np.all(np.abs(w - q * sc) <= 0.5 * sc * (1 + 1e-6))


def test_oracle_int8_hand_example():
    w = np.array([[31.75, -0.375, 0.125, 0.625, -31.75, 0.0]], np.float32)   # scale 0.25
    q, s = oq.quantize_int8_row(w)
    assert s[0] == 0.25
    assert list(q[0]) == [127, -2, 0, 2, -127, 0]
    q0, s0 = oq.quantize_int8_row(np.zeros((1, 4), np.float32))
    assert s0[0] == 0 and not q0.any()


# ---- library against the oracle -----------------------------------------------------------------

def _weights(seed, N, K):
    rng = np.random.default_rng(seed)
    w = rng.normal(0, 0.02, (N, K)).astype(np.float32)
    w[1, :128] = 0.0                                        # a zero group
    w[2] = 0.0                                              # a zero row
    w[3, :128] = np.float32(0.125) * rng.integers(-7, 8, 128)   # exact multiples and ties
    w[3, 0] = 0.875
    w[4, 5] = 1e-3                                          # one large value in a group
    return w


def test_library_int4_quantizer_matches_the_oracle(qd):
    w = _weights(1, 96, 1024)
    q, s = qd.quantize_int4(w)
    q0, s0 = oq.quantize_int4_g128(w)
    assert np.array_equal(s, s0)
    assert np.array_equal(q, q0)


def test_library_int8_quantizer_matches_the_oracle(qd):
    w = _weights(2, 64, 768)
    q, s = qd.quantize_int8(w)
    q0, s0 = oq.quantize_int8_row(w)
    assert np.array_equal(s.view(np.uint32), s0.view(np.uint32))
    assert np.array_equal(q, q0)


def test_quantizers_reject_bad_input(qd):
    from quantized_decode_gb300 import LLMError, _lib as L
    with pytest.raises(LLMError) as e:
        qd.quantize_int4(np.zeros((2, 100), np.float32))
    assert e.value.code == L.LLM_ERR_ARG
    w = np.zeros((2, 128), np.float32)
    w[1, 7] = np.nan
    for f in (qd.quantize_int4, qd.quantize_int8):
        with pytest.raises(LLMError) as e:
            f(w)
        assert e.value.code == L.LLM_ERR_ARG


# ---- the model file ---------------------------------------------------------------------------

TINY8 = sm.ModelConfig("tiny-int8", 2, 256, 4, 2, 64, 768, 1024, qkv_bias=False, qk_norm=True,
                       weight_format=sm.FMT_INT8_ROW, max_context=256)


def _cfg(name):
    return sm.CONFIGS["tiny"] if name == "tiny" else TINY8


def _expected_tensors(cfg, seed):
    """(name, bytes) in the documented file order, from the packer and the recipe."""
    from quantized_decode_gb300 import pack_int4, pack_int8
    int4 = cfg.weight_format == sm.FMT_INT4_G128
    get_proj, get_norms, embed, fnorm, lm = sm.recipe(cfg, seed)
    out = [("embed", np.ascontiguousarray(embed, np.uint16).tobytes()),
           ("final_norm", np.ascontiguousarray(fnorm, np.uint16).tobytes())]
    if not cfg.tied_lm_head:
        if lm["kind"] == "bf16":
            out.append(("lm_head", np.ascontiguousarray(lm["w"], np.uint16).tobytes()))
        else:
            out.append(("lm_head", pack_int8(lm["codes"]).tobytes()))
            out.append(("lm_scale", np.ascontiguousarray(lm["scales"], np.float32).tobytes()))
    for l in range(cfg.n_layers):
        for p in ("q", "k", "v", "o", "gate", "up", "down"):
            t = get_proj(l, p)
            out.append((f"{l}.w{p}", (pack_int4(t["codes"]) if int4 else pack_int8(t["codes"])).tobytes()))
            out.append((f"{l}.s{p}", np.ascontiguousarray(t["scales"]).tobytes()))
            if p in "qkv" and cfg.qkv_bias:
                out.append((f"{l}.b{p}", np.ascontiguousarray(t["bias"], np.uint16).tobytes()))
        n = get_norms(l)
        out.append((f"{l}.attn_norm", np.ascontiguousarray(n["attn_norm"], np.uint16).tobytes()))
        out.append((f"{l}.mlp_norm", np.ascontiguousarray(n["mlp_norm"], np.uint16).tobytes()))
        if cfg.qk_norm:
            out.append((f"{l}.q_norm", np.ascontiguousarray(n["q_norm"], np.uint16).tobytes()))
            out.append((f"{l}.k_norm", np.ascontiguousarray(n["k_norm"], np.uint16).tobytes()))
    return out


def _fnv1a64(b):
    h = 0xcbf29ce484222325
    for x in b:
        h = ((h ^ x) * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return h


def _write(qd, cfg, path, seed=5):
    qd.write_model_file(path, cfg, *sm.recipe(cfg, seed))
    return open(path, "rb").read()


@pytest.mark.parametrize("name", ["tiny", "tiny-int8"])
def test_file_follows_the_documented_map(qd, tmp_path, name):
    import struct
    cfg = _cfg(name)
    path = tmp_path / "m.qd"
    data = _write(qd, cfg, path)
    c = qd.make_config(cfg)
    n = ctypes.c_int64()
    assert qd.load().llm_model_file_bytes(ctypes.byref(c), ctypes.byref(n)) == 0
    assert len(data) == n.value
    assert data[:8] == b"QDECODEW"
    assert struct.unpack_from("<II", data, 8) == (1, 256)
    assert data[16:80] == bytes(c)
    poff, pbytes, csum = struct.unpack_from("<QQQ", data, 80)
    assert (poff, pbytes) == (256, len(data) - 256)
    assert csum == _fnv1a64(data[:96]) and not any(data[104:256])
    off = 256
    for tname, b in _expected_tensors(cfg, 5):
        at = (off + 127) // 128 * 128
        assert not any(data[off:at]), f"padding before {tname}"
        assert data[at:at + len(b)] == b, tname
        off = at + len(b)
    assert off == len(data)
    r = qd.read_model_config(path)
    assert bytes(r) == bytes(c)


def test_file_refusals(qd, tmp_path):
    import struct
    from quantized_decode_gb300 import LLMError, _lib as L
    cfg = sm.CONFIGS["tiny"]
    good = _write(qd, cfg, tmp_path / "g.qd")

    def code_of(blob):
        p = tmp_path / "x.qd"
        p.write_bytes(blob)
        with pytest.raises(LLMError) as e:
            qd.read_model_config(p)
        return e.value.code

    bad = bytearray(good)
    bad[0] ^= 1
    assert code_of(bytes(bad)) == L.LLM_ERR_FORMAT                       # magic
    bad = bytearray(good)
    bad[20] ^= 1
    assert code_of(bytes(bad)) == L.LLM_ERR_FORMAT                       # checksum
    assert code_of(good[:-1]) == L.LLM_ERR_FORMAT                        # truncated
    assert code_of(good[:100]) == L.LLM_ERR_FORMAT
    bad = bytearray(good)
    struct.pack_into("<I", bad, 8, 2)                                     # version
    struct.pack_into("<Q", bad, 96, _fnv1a64(bytes(bad[:96])))
    assert code_of(bytes(bad)) == L.LLM_ERR_FORMAT
    bad = bytearray(good)
    lid = L.llm_config.layout_id.offset
    struct.pack_into("<i", bad, 16 + lid, L.LLM_LAYOUT_INT8_ROW)          # layout id
    struct.pack_into("<Q", bad, 96, _fnv1a64(bytes(bad[:96])))
    assert code_of(bytes(bad)) == L.LLM_ERR_LAYOUT
    bad = bytearray(good)
    struct.pack_into("<i", bad, 16, 1 << 30)                              # n_layers: a crafted header
    struct.pack_into("<Q", bad, 96, _fnv1a64(bytes(bad[:96])))
    assert code_of(bytes(bad)) == L.LLM_ERR_FORMAT
    with pytest.raises(LLMError) as e:
        qd.read_model_config(tmp_path / "missing.qd")
    assert e.value.code == L.LLM_ERR_IO


def test_file_write_refusals(qd, tmp_path):
    from quantized_decode_gb300 import _lib as L
    lib = qd.load()
    cfg = qd.make_config(sm.CONFIGS["tiny"])
    layers = (L.llm_layer_weights * cfg.n_layers)()
    w = L.llm_weights()
    w.layers = layers
    p = str(tmp_path / "w.qd").encode()
    assert lib.llm_model_file_write(p, ctypes.byref(cfg), ctypes.byref(w)) == L.LLM_ERR_ARG   # null tensors
    cfg.layout_id = L.LLM_LAYOUT_INT8_ROW
    assert lib.llm_model_file_write(p, ctypes.byref(cfg), ctypes.byref(w)) == L.LLM_ERR_LAYOUT
    assert lib.llm_model_file_write(None, ctypes.byref(cfg), ctypes.byref(w)) == L.LLM_ERR_ARG
    h = ctypes.c_void_p()
    assert lib.llm_create_from_file(str(tmp_path / "missing.qd").encode(), 0, None,
                                    ctypes.byref(h)) == L.LLM_ERR_IO
    assert not h.value
