"""CPU oracle for the batch-1 quantized decode step (ctypes binding of oracle.c).

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's CPU
baseline leg may import this package.  The engine never does; the two share no code.

Two precisions of the same C source: ``Oracle("f32")`` is the FP32 decoder the
acceptance criterion names, ``Oracle("f64")`` runs the same steps in double and bounds
the fp32 variant's own rounding.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_INT4_G128 = 1
FMT_INT8_ROW = 2


def build(force=False):
    """Compile oracle.c twice (fp32 and fp64 arithmetic) into liboracle.so."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        o32, o64 = tmp + ".f32.o", tmp + ".f64.o"
        common = ["gcc", "-O3", "-fopenmp", "-fPIC", "-ffp-contract=off", "-c", _SRC]
        subprocess.check_call(common + ["-o", o32])
        subprocess.check_call(common + ["-DOR_REAL=double", "-DOR_DOUBLE_BUILD", "-o", o64])
        subprocess.check_call(["gcc", "-shared", "-fopenmp", "-o", tmp, o32, o64, "-lm"])
        os.remove(o32)
        os.remove(o64)
        os.replace(tmp, _SO)
    return _SO


class OrConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "mlp", "vocab")] + \
               [("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float)] + \
               [(n, ctypes.c_int32) for n in
                ("qkv_bias", "qk_norm", "tied_lm_head", "weight_format")]


_LAYER_FIELDS = ("wq", "sq", "bq", "wk", "sk", "bk", "wv", "sv", "bv", "wo", "so", "wg", "sg",
                 "wu", "su", "wd", "sd", "attn_norm", "mlp_norm", "q_norm", "k_norm")


class OrLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _LAYER_FIELDS]


class OrWeights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("lm_scale", ctypes.c_void_p),
                ("layers", ctypes.POINTER(OrLayer))]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int32
            lib.or_pack_int4.argtypes = [vp, i64, i64, vp]
            lib.or_pack_int4.restype = None
            lib.or_unpack_int4.argtypes = [vp, i64, i64, vp]
            lib.or_unpack_int4.restype = None
            lib.or_bf16_round.argtypes = [f32]
            lib.or_bf16_round.restype = ctypes.c_uint16
            lib.or_argmax.argtypes = [vp, i64]
            lib.or_argmax.restype = i64
            lib.or_threads.argtypes = []
            lib.or_threads.restype = ctypes.c_int
            lib.or_set_threads.argtypes = [ctypes.c_int]
            lib.or_set_threads.restype = None
            for p in ("f32", "f64"):
                g = lambda n: getattr(lib, f"or_{p}_{n}")  # noqa: E731
                g("rmsnorm").argtypes = [vp, vp, i64, f32, vp]
                g("rope").argtypes = [vp, i64, i64, i64, ctypes.c_double]
                g("softmax").argtypes = [vp, i64, vp]
                g("silu_mul").argtypes = [vp, vp, i64, vp]
                g("gemv_int4").argtypes = [vp, vp, vp, i64, i64, vp, vp, vp]
                g("gemv_int8").argtypes = [vp, vp, i64, i64, vp, vp, vp]
                g("gemv_bf16").argtypes = [vp, i64, i64, vp, vp, vp]
                g("attention").argtypes = [vp, vp, vp, i64, i64, i64, i64, vp]
                g("step").argtypes = [ctypes.POINTER(OrConfig), ctypes.POINTER(OrWeights), vp, vp,
                                      i64, i32, i64, vp, vp]
                g("step").restype = ctypes.c_int
                g("prefill").argtypes = [ctypes.POINTER(OrConfig), ctypes.POINTER(OrWeights), vp, vp,
                                         i64, vp, i64, i64, vp]
                g("prefill").restype = ctypes.c_int
                for n in ("rmsnorm", "rope", "softmax", "silu_mul", "gemv_int4", "gemv_int8",
                          "gemv_bf16", "attention"):
                    g(n).restype = None
            _lib = lib
    return _lib


def threads():
    """Host threads the oracle's parallel loops use."""
    return int(_load().or_threads())


def set_threads(n):
    """Set the oracle's host threads (timing only: its results do not depend on them)."""
    _load().or_set_threads(int(n))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- integer work

def pack_int4(codes):
    """Logical codes [N][K] in [-8,7] -> ValueShuffle words [N][K/8] (uint32)."""
    codes = _c(codes, np.int8)
    N, K = codes.shape
    out = np.empty((N, K // 8), dtype=np.uint32)
    _load().or_pack_int4(_p(codes), N, K, _p(out))
    return out


def unpack_int4(words, K=None):
    words = _c(words, np.uint32)
    N = words.shape[0]
    K = words.shape[1] * 8 if K is None else K
    out = np.empty((N, K), dtype=np.int8)
    _load().or_unpack_int4(_p(words), N, K, _p(out))
    return out


def bf16_round(x):
    """fp32 -> bfloat16 bits, round to nearest even (the KV cache's storage rounding)."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    return np.array([lib.or_bf16_round(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def argmax(v):
    v = _c(v, np.float32)
    return int(_load().or_argmax(_p(v), v.size))


# ---------------------------------------------------------------- floating-point work

class Oracle:
    def __init__(self, precision="f32"):
        assert precision in ("f32", "f64")
        self.precision = precision
        self.dtype = np.float32 if precision == "f32" else np.float64
        self._lib = _load()

    def _f(self, name):
        return getattr(self._lib, f"or_{self.precision}_{name}")

    def rmsnorm(self, x, gamma_bf16, eps):
        x = _c(x, self.dtype)
        g = _c(gamma_bf16, np.uint16)
        y = np.empty_like(x)
        self._f("rmsnorm")(_p(x), _p(g), x.size, eps, _p(y))
        return y

    def rope(self, v, n_heads, d, pos, base):
        v = _c(v, self.dtype).copy()
        self._f("rope")(_p(v), n_heads, d, pos, base)
        return v

    def softmax(self, s):
        s = _c(s, self.dtype)
        p = np.empty_like(s)
        self._f("softmax")(_p(s), s.size, _p(p))
        return p

    def silu_mul(self, g, u):
        g, u = _c(g, self.dtype), _c(u, self.dtype)
        out = np.empty_like(g)
        self._f("silu_mul")(_p(g), _p(u), g.size, _p(out))
        return out

    def gemv_int4(self, words, scales, x, bias=None):
        """y = dequant(words, scales) @ x (+ bias); also returns sum_k |W_nk x_k|."""
        words, scales = _c(words, np.uint32), _c(scales, np.uint16)
        x = _c(x, self.dtype)
        N, K = words.shape[0], words.shape[1] * 8
        assert x.size == K and scales.shape == (N, K // 128)
        b = None if bias is None else _c(bias, np.uint16)
        y = np.empty(N, self.dtype)
        a = np.empty(N, self.dtype)
        self._f("gemv_int4")(_p(words), _p(scales), _p(b), N, K, _p(x), _p(y), _p(a))
        return y, a

    def gemv_int8(self, codes, scales, x):
        codes, scales, x = _c(codes, np.int8), _c(scales, np.float32), _c(x, self.dtype)
        N, K = codes.shape
        y = np.empty(N, self.dtype)
        a = np.empty(N, self.dtype)
        self._f("gemv_int8")(_p(codes), _p(scales), N, K, _p(x), _p(y), _p(a))
        return y, a

    def gemv_bf16(self, w, x):
        w, x = _c(w, np.uint16), _c(x, self.dtype)
        N, K = w.shape
        y = np.empty(N, self.dtype)
        a = np.empty(N, self.dtype)
        self._f("gemv_bf16")(_p(w), N, K, _p(x), _p(y), _p(a))
        return y, a

    def attention(self, q, k_cache, v_cache, Hq, Hkv, d):
        """q [Hq*d]; k_cache, v_cache bf16 bits [T][Hkv][d] -> out [Hq*d]."""
        q = _c(q, self.dtype)
        kc, vc = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
        T = kc.shape[0]
        out = np.empty(Hq * d, self.dtype)
        self._f("attention")(_p(q), _p(kc), _p(vc), T, Hq, Hkv, d, _p(out))
        return out


class OracleModel:
    """A decoder held in host memory in the oracle's own packed form.

    Built from the logical tensors of synth.model (codes, scales, gains, biases); INT4
    codes are packed with the oracle's own packer.  Holds its own KV cache.
    """

    def __init__(self, cfg, seed, precision="f32", t_max=None, tensors=None, norms=None,
                 embed=None, lm_head=None):
        """tensors(layer, proj) / norms(layer) / embed [V][h] / lm_head (synth.model.lm_head's
        dict) override the seeded draws (the model-level pins build structured special cases
        through them; the full-depth tests pass arrays already drawn)."""
        from synth import model as sm
        self.cfg = cfg
        self.seed = seed
        self.oracle = Oracle(precision)
        self.t_max = t_max or cfg.max_context
        self._keep = []
        c = OrConfig(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                     cfg.mlp, cfg.vocab, cfg.rms_eps, cfg.rope_base, int(cfg.qkv_bias),
                     int(cfg.qk_norm), int(cfg.tied_lm_head), cfg.weight_format)
        self.c = c
        layers = (OrLayer * cfg.n_layers)()
        names = {"q": ("wq", "sq", "bq"), "k": ("wk", "sk", "bk"), "v": ("wv", "sv", "bv"),
                 "o": ("wo", "so", None), "gate": ("wg", "sg", None), "up": ("wu", "su", None),
                 "down": ("wd", "sd", None)}
        for l in range(cfg.n_layers):
            for proj in sm.PROJS:
                t = tensors(l, proj) if tensors else sm.layer_proj(cfg, seed, l, proj)
                w = pack_int4(t["codes"]) if cfg.weight_format == FMT_INT4_G128 else \
                    _c(t["codes"], np.int8)
                s = _c(t["scales"], np.uint16 if cfg.weight_format == FMT_INT4_G128 else np.float32)
                fw, fs, fb = names[proj]
                setattr(layers[l], fw, self._hold(w))
                setattr(layers[l], fs, self._hold(s))
                if fb and t["bias"] is not None:
                    setattr(layers[l], fb, self._hold(_c(t["bias"], np.uint16)))
            nl = norms(l) if norms else sm.layer_norms(cfg, seed, l)
            for k, v in nl.items():
                if v is not None:
                    setattr(layers[l], k, self._hold(_c(v, np.uint16)))
        self.layers = layers
        self.embed = _c(sm.embedding(cfg, seed) if embed is None else embed, np.uint16)
        lm = sm.lm_head(cfg, seed) if lm_head is None else lm_head
        w = OrWeights()
        w.embed = self._hold(self.embed)
        w.final_norm = self._hold(_c(sm.final_norm(cfg, seed), np.uint16))
        if lm["kind"] == "tied":
            w.lm_head = w.embed
            w.lm_scale = None
        elif lm["kind"] == "bf16":
            w.lm_head = self._hold(_c(lm["w"], np.uint16))
            w.lm_scale = None
        else:
            w.lm_head = self._hold(_c(lm["codes"], np.int8))
            w.lm_scale = self._hold(_c(lm["scales"], np.float32))
        w.layers = layers
        self.w = w
        shape = (cfg.n_layers, self.t_max, cfg.n_kv_heads, cfg.head_dim)
        self.k_cache = np.zeros(shape, np.uint16)
        self.v_cache = np.zeros(shape, np.uint16)

    def _hold(self, a):
        self._keep.append(a)
        return a.ctypes.data_as(ctypes.c_void_p)

    def step(self, token, pos, want_hidden=False):
        """One decode step; returns logits (fp32) [and the final residual]."""
        cfg = self.cfg
        logits = np.empty(cfg.vocab, np.float32)
        hidden = np.empty(cfg.hidden, np.float32) if want_hidden else None
        rc = self.oracle._f("step")(ctypes.byref(self.c), ctypes.byref(self.w), _p(self.k_cache),
                                    _p(self.v_cache), self.t_max, int(token), int(pos),
                                    _p(logits), _p(hidden))
        if rc != 0:
            raise ValueError(f"oracle step rejected token={token} pos={pos}")
        return (logits, hidden) if want_hidden else logits

    def prefill(self, tokens, pos0=0):
        """The step applied to tokens at positions pos0.. (every linear layer evaluated for
        all rows at once, each output the same sum as the step's); returns the logits of the
        last token (fp32).  Equals len(tokens) calls of step() bit for bit."""
        cfg = self.cfg
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        logits = np.empty(cfg.vocab, np.float32)
        rc = self.oracle._f("prefill")(ctypes.byref(self.c), ctypes.byref(self.w), _p(self.k_cache),
                                       _p(self.v_cache), self.t_max, _p(toks), toks.size, int(pos0),
                                       _p(logits))
        if rc != 0:
            raise ValueError(f"oracle prefill rejected n={toks.size} pos0={pos0}")
        return logits

    def set_kv(self, layer, k, v, start=0):
        """Write bf16 K/V rows [T][Hkv][d] at positions start.. of one layer."""
        T = k.shape[0]
        self.k_cache[layer, start:start + T] = k
        self.v_cache[layer, start:start + T] = v
