"""Python face of the C ABI: an Engine handle and a device-resident packed model.

PyTorch supplies device memory and the stream; packing runs in libllm.so's host packer and
every step of decoding runs in libllm.so's CUDA kernels.
"""
import ctypes

import numpy as np

from . import _lib as L

PROJ_FIELDS = {"q": ("wq", "sq", "bq"), "k": ("wk", "sk", "bk"), "v": ("wv", "sv", "bv"),
               "o": ("wo", "so", None), "gate": ("wg", "sg", None), "up": ("wu", "su", None),
               "down": ("wd", "sd", None)}
PROJS = ("q", "k", "v", "o", "gate", "up", "down")


def _np_ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def pack_int4(codes):
    """Logical INT4 codes [N][K] (int8, [-8,7]) -> ValueShuffle words [N][K/8] via libllm."""
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    N, K = codes.shape
    words = np.empty((N, K // 8), dtype=np.uint32)
    L.check(L.load().llm_pack_int4_g128(_np_ptr(codes), N, K, _np_ptr(words)), "llm_pack_int4_g128")
    return words


def pack_int8(codes):
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    out = np.empty_like(codes)
    L.check(L.load().llm_pack_int8_row(_np_ptr(codes), codes.shape[0], codes.shape[1], _np_ptr(out)),
            "llm_pack_int8_row")
    return out


def make_config(cfg):
    """llm_config from any object with the model-shape attributes."""
    fmt = int(cfg.weight_format)
    return L.llm_config(
        n_layers=cfg.n_layers, hidden=cfg.hidden, n_q_heads=cfg.n_q_heads,
        n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, mlp=cfg.mlp, vocab=cfg.vocab,
        rms_eps=cfg.rms_eps, rope_base=cfg.rope_base, qkv_bias=int(cfg.qkv_bias),
        qk_norm=int(cfg.qk_norm), tied_lm_head=int(cfg.tied_lm_head), weight_format=fmt,
        layout_id=L.LLM_LAYOUT_INT4_VALUESHUFFLE if fmt == L.LLM_FMT_INT4_G128 else L.LLM_LAYOUT_INT8_ROW,
        max_context=cfg.max_context, page_tokens=16)


def quantize_int4(w):
    """fp32 weights [N][K] -> (codes int8 [N][K], bf16 scale bits [N][K/128]) by libllm's
    absmax/7 group-128 quantizer (llm_quantize_int4_g128)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    codes = np.empty((N, K), dtype=np.int8)
    scales = np.empty((N, K // 128), dtype=np.uint16)
    L.check(L.load().llm_quantize_int4_g128(_np_ptr(w), N, K, _np_ptr(codes), _np_ptr(scales)),
            "llm_quantize_int4_g128")
    return codes, scales


def quantize_int8(w):
    """fp32 weights [N][K] -> (codes int8 [N][K], fp32 row scales [N]) (llm_quantize_int8_row)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    codes = np.empty((N, K), dtype=np.int8)
    scales = np.empty(N, dtype=np.float32)
    L.check(L.load().llm_quantize_int8_row(_np_ptr(w), N, K, _np_ptr(codes), _np_ptr(scales)),
            "llm_quantize_int8_row")
    return codes, scales


def _fill(cfg, get_proj, get_norms, embed, final_norm, lm_head, put):
    """llm_layer_weights array and llm_weights with every tensor passed through put(array)
    -> pointer (device upload, or a host array kept alive)."""
    int4 = int(cfg.weight_format) == L.LLM_FMT_INT4_G128
    layers = (L.llm_layer_weights * cfg.n_layers)()
    for l in range(cfg.n_layers):
        for proj in PROJS:
            t = get_proj(l, proj)
            fw, fs, fb = PROJ_FIELDS[proj]
            w = pack_int4(t["codes"]) if int4 else pack_int8(t["codes"])
            setattr(layers[l], fw, put(w))
            setattr(layers[l], fs, put(np.ascontiguousarray(t["scales"])))
            if fb and t.get("bias") is not None:
                setattr(layers[l], fb, put(np.ascontiguousarray(t["bias"], dtype=np.uint16)))
        for k, v in get_norms(l).items():
            if v is not None:
                setattr(layers[l], k, put(np.ascontiguousarray(v, dtype=np.uint16)))
    w = L.llm_weights()
    w.embed = put(np.ascontiguousarray(embed, dtype=np.uint16))
    w.final_norm = put(np.ascontiguousarray(final_norm, dtype=np.uint16))
    if lm_head["kind"] == "bf16":
        w.lm_head = put(np.ascontiguousarray(lm_head["w"], dtype=np.uint16))
    elif lm_head["kind"] == "int8":
        w.lm_head = put(pack_int8(lm_head["codes"]))
        w.lm_scale = put(np.ascontiguousarray(lm_head["scales"], dtype=np.float32))
    w.layers = layers
    return layers, w


class DeviceModel:
    """Packed decoder weights resident in device memory (torch tensors) + the ABI structs.

    get_proj(layer, proj) -> dict(codes [N][K] int8, scales, bias or None)
    get_norms(layer) -> dict(attn_norm, mlp_norm, q_norm, k_norm) of bf16 bit arrays or None
    embed: bf16 bits [V][h]; final_norm: bf16 bits [h];
    lm_head: dict(kind='tied'|'bf16'|'int8', w | codes+scales)
    """

    def __init__(self, cfg, get_proj, get_norms, embed, final_norm, lm_head, device="cuda"):
        import torch
        self.cfg = cfg
        self.device = device
        self._t = []

        def up(a):
            a = np.ascontiguousarray(a)
            t = torch.from_numpy(a.view(np.uint8).reshape(-1)).to(device)
            self._t.append(t)
            return t.data_ptr()

        self.layers, self.weights = _fill(cfg, get_proj, get_norms, embed, final_norm, lm_head, up)

    def nbytes(self):
        return sum(t.numel() for t in self._t)


def write_model_file(path, cfg, get_proj, get_norms, embed, final_norm, lm_head):
    """Pack a model (same arguments as DeviceModel) and write it as one model file
    (llm_model_file_write); no GPU needed."""
    keep = []

    def host(a):
        a = np.ascontiguousarray(a)
        keep.append(a)
        return a.ctypes.data

    layers, w = _fill(cfg, get_proj, get_norms, embed, final_norm, lm_head, host)
    c = make_config(cfg)
    L.check(L.load().llm_model_file_write(str(path).encode(), ctypes.byref(c), ctypes.byref(w)),
            "llm_model_file_write")
    del layers, keep


def read_model_config(path):
    """The llm_config in a model file's header (checked; no weights read)."""
    c = L.llm_config()
    L.check(L.load().llm_model_file_read_config(str(path).encode(), ctypes.byref(c)),
            "llm_model_file_read_config")
    return c


class Engine:
    """One decode sequence on one GPU (llm_t handle)."""

    def __init__(self, model, stream=None, config=None):
        self.lib = L.load()
        self.model = model
        self.cfg = config if config is not None else make_config(model.cfg)
        self.vocab = self.cfg.vocab
        h = ctypes.c_void_p()
        s = None if stream is None else ctypes.c_void_p(stream)
        L.check(self.lib.llm_create(ctypes.byref(self.cfg), ctypes.byref(model.weights), s,
                                    ctypes.byref(h)), "llm_create")
        self.h = h

    @classmethod
    def from_file(cls, path, max_context=0, stream=None):
        """An engine on a model file's weights (llm_create_from_file; the handle owns their
        device copy).  max_context > 0 overrides the file's."""
        self = cls.__new__(cls)
        self.lib = L.load()
        self.model = None
        self.cfg = read_model_config(path)
        if max_context > 0:
            self.cfg.max_context = max_context
        self.vocab = self.cfg.vocab
        h = ctypes.c_void_p()
        s = None if stream is None else ctypes.c_void_p(stream)
        self.h = None
        L.check(self.lib.llm_create_from_file(str(path).encode(), max_context, s, ctypes.byref(h)),
                "llm_create_from_file")
        self.h = h
        return self

    def close(self):
        if self.h:
            self.lib.llm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, tokens):
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        out = ctypes.c_int32()
        L.check(self.lib.llm_prefill(self.h, toks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                     toks.size, ctypes.byref(out)), "llm_prefill")
        return out.value

    def decode_step(self, forced=-1):
        out = ctypes.c_int32()
        L.check(self.lib.llm_decode_step(self.h, int(forced), ctypes.byref(out)), "llm_decode_step")
        return out.value

    def decode_enqueue(self, n):
        L.check(self.lib.llm_decode_enqueue(self.h, int(n)), "llm_decode_enqueue")

    def sync(self):
        L.check(self.lib.llm_sync(self.h), "llm_sync")

    def last_token(self):
        out = ctypes.c_int32()
        L.check(self.lib.llm_last_token(self.h, ctypes.byref(out)), "llm_last_token")
        return out.value

    def logits(self):
        out = np.empty(self.vocab, dtype=np.float32)
        L.check(self.lib.llm_logits(self.h, _np_ptr(out), self.vocab), "llm_logits")
        return out

    def seq_len(self):
        out = ctypes.c_int32()
        L.check(self.lib.llm_seq_len(self.h, ctypes.byref(out)), "llm_seq_len")
        return out.value

    def reset(self):
        L.check(self.lib.llm_reset(self.h), "llm_reset")

    def truncate(self, n):
        L.check(self.lib.llm_truncate(self.h, int(n)), "llm_truncate")

    def profile_step(self):
        """One greedy step timed per region (qkv, attention, o_proj, gate_up, down per layer, then
        lm_head) -> array of ms (5L + 1)."""
        n_layers = self.cfg.n_layers
        out = np.empty(5 * n_layers + 1, dtype=np.float32)
        n = ctypes.c_int32()
        L.check(self.lib.llm_profile_step(self.h, _np_ptr(out), out.size, ctypes.byref(n)),
                "llm_profile_step")
        return out[:n.value]

    def timeline_steps(self, n_steps):
        """n_steps greedy steps replayed from one graph whose launches record their last CTA's
        finish time (llm_timeline_steps) -> uint64 ns array [n_steps][launches per step]."""
        per = 5 * self.cfg.n_layers + 2
        out = np.zeros(n_steps * per, dtype=np.uint64)
        n = ctypes.c_int32()
        L.check(self.lib.llm_timeline_steps(self.h, int(n_steps), _np_ptr(out), out.size, ctypes.byref(n)),
                "llm_timeline_steps")
        return out[:n_steps * n.value].reshape(n_steps, n.value)

    def set_pdl(self, on):
        L.check(self.lib.llm_set_pdl(self.h, int(bool(on))), "llm_set_pdl")

    def set_sampling(self, temperature, top_k=1, top_p=1.0, seed=0):
        """temperature <= 0: greedy argmax (default); otherwise top-k / top-p sampling on the GPU."""
        L.check(self.lib.llm_set_sampling(self.h, float(temperature), int(top_k), float(top_p), int(seed)),
                "llm_set_sampling")

    def set_act_int8(self, on):
        L.check(self.lib.llm_set_act_int8(self.h, int(on)), "llm_set_act_int8")

    def set_fused_attention(self, on):
        """True: QKV projection and attention of a layer in one kernel (where the model fits it)."""
        L.check(self.lib.llm_set_fused_attention(self.h, int(bool(on))), "llm_set_fused_attention")

    def set_persistent(self, on):
        """True: the step is the persistent whole-step kernel; False: the kernel chain."""
        L.check(self.lib.llm_set_persistent(self.h, int(bool(on))), "llm_set_persistent")

    def debug_step_wait(self, extra_arrivals, counter_wait_ns):
        """Test hook: the persistent kernel's phase-counter waits expect extra_arrivals (0/1)
        more arrivals and give up after counter_wait_ns (llm_debug_step_wait)."""
        L.check(self.lib.llm_debug_step_wait(self.h, int(extra_arrivals), int(counter_wait_ns)),
                "llm_debug_step_wait")

    def set_o_fold(self, on):
        """True: o_proj inside the decode attention clusters; False (default): its own GEMV."""
        L.check(self.lib.llm_set_o_fold(self.h, int(bool(on))), "llm_set_o_fold")

    def o_fold(self):
        """The current set_o_fold setting."""
        out = ctypes.c_int32()
        L.check(self.lib.llm_get_o_fold(self.h, ctypes.byref(out)), "llm_get_o_fold")
        return bool(out.value)

    def set_fused_mlp(self, on):
        """True (default where it fits): the MLP block as one kernel; False: gate/up + down."""
        L.check(self.lib.llm_set_fused_mlp(self.h, int(bool(on))), "llm_set_fused_mlp")

    def step_kinds(self):
        """Names of the launches of one decode step, in order (empty for the persistent kernel)."""
        out = np.zeros(5 * self.cfg.n_layers + 2, dtype=np.int32)
        n = ctypes.c_int32()
        L.check(self.lib.llm_step_kinds(self.h, _np_ptr(out), out.size, ctypes.byref(n)), "llm_step_kinds")
        return [L.KIND_NAMES[k] for k in out[:n.value]]

    def set_l2_prefetch(self, flags):
        """Bulk L2 prefetch of later kernels' weights (llm_set_l2_prefetch flags; 0 = off)."""
        L.check(self.lib.llm_set_l2_prefetch(self.h, int(flags)), "llm_set_l2_prefetch")

    def set_prefill_batched(self, on):
        """True: prompts run as one batch on the tensor cores; False: token by token."""
        L.check(self.lib.llm_set_prefill_batched(self.h, int(bool(on))), "llm_set_prefill_batched")

    def set_graph_mode(self, on):
        L.check(self.lib.llm_set_graph_mode(self.h, int(bool(on))), "llm_set_graph_mode")

    def debug_kv(self, set_len=-1):
        """-> (k_pool ptr, v_pool ptr, page_table ptr, n_pages)."""
        k, v, pt, n = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_int32()
        L.check(self.lib.llm_debug_kv(self.h, ctypes.byref(k), ctypes.byref(v), ctypes.byref(pt),
                                      ctypes.byref(n), int(set_len)), "llm_debug_kv")
        return k.value, v.value, pt.value, n.value


class BatchEngine:
    """Up to 8 sequences decoding together over one paged K/V pool (llm_batch_t handle)."""

    def __init__(self, model, max_seqs, n_pages=0, stream=None, config=None):
        self.lib = L.load()
        self.model = model
        self.cfg = config if config is not None else make_config(model.cfg)
        self.vocab = self.cfg.vocab
        h = ctypes.c_void_p()
        s = None if stream is None else ctypes.c_void_p(stream)
        L.check(self.lib.llm_batch_create(ctypes.byref(self.cfg), ctypes.byref(model.weights), int(max_seqs),
                                          int(n_pages), s, ctypes.byref(h)), "llm_batch_create")
        self.h = h

    def close(self):
        if self.h:
            self.lib.llm_batch_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self):
        out = ctypes.c_int32()
        L.check(self.lib.llm_batch_add(self.h, ctypes.byref(out)), "llm_batch_add")
        return out.value

    def release(self, seq):
        L.check(self.lib.llm_batch_release(self.h, int(seq)), "llm_batch_release")

    def step(self, seqs, inputs=None):
        """One step for the sequences seqs; inputs (same length; -1 = the previous token) or None."""
        sq = np.ascontiguousarray(seqs, dtype=np.int32)
        inp = None if inputs is None else np.ascontiguousarray(inputs, dtype=np.int32)
        out = np.empty(sq.size, dtype=np.int32)
        L.check(self.lib.llm_batch_step(self.h, _np_ptr(sq), None if inp is None else _np_ptr(inp), sq.size,
                                        _np_ptr(out)), "llm_batch_step")
        return out

    def prefill(self, seq, tokens):
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        out = ctypes.c_int32()
        L.check(self.lib.llm_batch_prefill(self.h, int(seq), _np_ptr(toks), toks.size, ctypes.byref(out)),
                "llm_batch_prefill")
        return out.value

    def logits(self, seq):
        out = np.empty(self.vocab, dtype=np.float32)
        L.check(self.lib.llm_batch_logits(self.h, int(seq), _np_ptr(out), self.vocab), "llm_batch_logits")
        return out

    def seq_info(self, seq):
        """-> (length, physical pages in logical order, free pages left)."""
        n, np_, free = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        L.check(self.lib.llm_batch_seq_info(self.h, int(seq), ctypes.byref(n), None, 0, ctypes.byref(np_),
                                            ctypes.byref(free)), "llm_batch_seq_info")
        pages = np.empty(max(np_.value, 1), dtype=np.int32)
        L.check(self.lib.llm_batch_seq_info(self.h, int(seq), None, _np_ptr(pages), pages.size, None, None),
                "llm_batch_seq_info")
        return n.value, pages[:np_.value], free.value

    def set_page_order(self, order):
        o = np.ascontiguousarray(order, dtype=np.int32)
        L.check(self.lib.llm_batch_set_page_order(self.h, _np_ptr(o), o.size), "llm_batch_set_page_order")

    def debug_kv(self):
        k, v, n = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_int32()
        L.check(self.lib.llm_batch_debug_kv(self.h, ctypes.byref(k), ctypes.byref(v), ctypes.byref(n)),
                "llm_batch_debug_kv")
        return k.value, v.value, n.value
