"""Checkpoint conversion (CPU): a synthetic safetensors checkpoint in two shards is converted,
and every tensor of the model file must equal the oracle's quantization of the source (packed
by the library's packer, which test_abi_host pins against the oracle's) or the source's bf16
bits, in the documented order."""
import json

import numpy as np
import pytest

from oracle import quantize as oq


def _write_safetensors(path, tensors):
    header, blobs, off = {}, [], 0
    for name, a in tensors.items():
        dt = {np.dtype(np.float32): "F32", np.dtype(np.uint16): "BF16"}[a.dtype]
        b = np.ascontiguousarray(a).tobytes()
        header[name] = {"dtype": dt, "shape": list(a.shape), "data_offsets": [off, off + len(b)]}
        blobs.append(b)
        off += len(b)
    h = json.dumps(header).encode()
    with open(path, "wb") as f:
        f.write(len(h).to_bytes(8, "little"))
        f.write(h)
        for b in blobs:
            f.write(b)


def _checkpoint(tmp_path, qwen3, tied):
    rng = np.random.default_rng(7)
    L, h, H, Hkv, d, F, V = 2, 256, 4, 2, 64, 768, 1024
    cfg = {"model_type": "qwen3" if qwen3 else "qwen2", "num_hidden_layers": L, "hidden_size": h,
           "num_attention_heads": H, "num_key_value_heads": Hkv, "head_dim": d, "intermediate_size": F,
           "vocab_size": V, "rms_norm_eps": 1e-6, "rope_theta": 1e6, "tie_word_embeddings": tied}
    (tmp_path / "config.json").write_text(json.dumps(cfg))

    def bf(*shape, std=0.02):
        return oq.bf16_rne_bits(rng.normal(0, std, shape).astype(np.float32))

    t = {"model.embed_tokens.weight": bf(V, h), "model.norm.weight": bf(h, std=1.0)}
    if not tied:
        t["lm_head.weight"] = rng.normal(0, 0.02, (V, h)).astype(np.float32)   # an fp32 tensor too
    for l in range(L):
        p = f"model.layers.{l}."
        for n, shape in (("self_attn.q_proj", (H * d, h)), ("self_attn.k_proj", (Hkv * d, h)),
                         ("self_attn.v_proj", (Hkv * d, h)), ("self_attn.o_proj", (h, H * d)),
                         ("mlp.gate_proj", (F, h)), ("mlp.up_proj", (F, h)), ("mlp.down_proj", (h, F))):
            t[p + n + ".weight"] = bf(*shape)
            if not qwen3 and n.split(".")[1] in ("q_proj", "k_proj", "v_proj"):
                t[p + n + ".bias"] = bf(shape[0])
        t[p + "input_layernorm.weight"] = bf(h, std=1.0)
        t[p + "post_attention_layernorm.weight"] = bf(h, std=1.0)
        if qwen3:
            t[p + "self_attn.q_norm.weight"] = bf(d, std=1.0)
            t[p + "self_attn.k_norm.weight"] = bf(d, std=1.0)
    names = sorted(t)
    half = len(names) // 2
    _write_safetensors(tmp_path / "model-00001-of-00002.safetensors", {n: t[n] for n in names[:half]})
    _write_safetensors(tmp_path / "model-00002-of-00002.safetensors", {n: t[n] for n in names[half:]})
    return cfg, t


def _f32(a):
    return (a.astype(np.uint32) << 16).view(np.float32) if a.dtype == np.uint16 else a


@pytest.mark.parametrize("qwen3,tied,int8", [(False, False, False), (False, True, False), (True, False, True)],
                         ids=["qwen2-int4", "qwen2-tied-int4", "qwen3-int8"])
def test_converted_file_holds_the_quantized_checkpoint(tmp_path, qwen3, tied, int8):
    import quantized_decode_gb300 as qd
    from quantized_decode_gb300 import convert as cv
    qd.build()
    cj, t = _checkpoint(tmp_path, qwen3, tied)
    out = tmp_path / "m.qd"
    cv.convert(str(tmp_path), str(out), int8=int8, max_context=512)
    c = qd.read_model_config(out)
    assert (c.n_layers, c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim, c.mlp, c.vocab) == \
        (2, 256, 4, 2, 64, 768, 1024)
    assert (c.qkv_bias, c.qk_norm, c.tied_lm_head, c.max_context) == (int(not qwen3), int(qwen3), int(tied), 512)
    assert c.weight_format == (2 if int8 else 1)

    def q(name):
        w = _f32(t[name])
        if int8:
            codes, s = oq.quantize_int8_row(w)
            return [qd.pack_int8(codes).tobytes(), s.tobytes()]
        codes, s = oq.quantize_int4_g128(w)
        return [qd.pack_int4(codes).tobytes(), s.tobytes()]

    want = [t["model.embed_tokens.weight"].tobytes(), t["model.norm.weight"].tobytes()]
    if not tied:
        if int8:
            want += q("lm_head.weight")
        else:
            want.append(oq.bf16_rne_bits(t["lm_head.weight"]).tobytes())
    for l in range(2):
        p = f"model.layers.{l}."
        for n in ("self_attn.q_proj", "self_attn.k_proj", "self_attn.v_proj", "self_attn.o_proj",
                  "mlp.gate_proj", "mlp.up_proj", "mlp.down_proj"):
            want += q(p + n + ".weight")
            if not qwen3 and n.endswith(("q_proj", "k_proj", "v_proj")):
                want.append(t[p + n + ".bias"].tobytes())
        want += [t[p + "input_layernorm.weight"].tobytes(), t[p + "post_attention_layernorm.weight"].tobytes()]
        if qwen3:
            want += [t[p + "self_attn.q_norm.weight"].tobytes(), t[p + "self_attn.k_norm.weight"].tobytes()]
    data = out.read_bytes()
    off = 256
    for i, b in enumerate(want):
        at = (off + 127) // 128 * 128
        assert data[at:at + len(b)] == b, i
        off = at + len(b)
    assert off == len(data)


def test_reader_rejects_unsupported_dtypes(tmp_path):
    from quantized_decode_gb300 import convert as cv
    p = tmp_path / "x.safetensors"
    h = json.dumps({"a": {"dtype": "I64", "shape": [1], "data_offsets": [0, 8]}}).encode()
    p.write_bytes(len(h).to_bytes(8, "little") + h + bytes(8))
    with pytest.raises(ValueError):
        cv.read_safetensors(str(p))
