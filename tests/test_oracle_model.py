"""Model-level pins of the oracle's composed decoder step (CPU only).

The composed step has no printed worked example on the pages, so it is pinned by
invariants that any correct decoder satisfies and that a plausible composition slip
breaks: the head-to-KV-group map, q/k versus v roles, the orientation of the down
projection, causality, the fp32 variant's rounding against the fp64 variant; and by
structured special cases: which matrix sits inside Swish, which norm feeds which block,
each residual added once, and a model whose whole step reduces to a closed form.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import model as sm

SEED = 1234
TINY = sm.CONFIGS["tiny"].with_(max_context=64)


def _gen(cfg, seed=SEED):
    return lambda l, p: sm.layer_proj(cfg, seed, l, p)


def _run(model, tokens):
    out = []
    for pos, t in enumerate(tokens):
        out.append(model.step(int(t), pos))
    return out


def test_step_is_deterministic_and_finite():
    m1 = oracle.OracleModel(TINY, SEED)
    m2 = oracle.OracleModel(TINY, SEED)
    toks = sm.prompt(TINY, SEED, 6)
    a, b = _run(m1, toks), _run(m2, toks)
    for x, y in zip(a, b):
        assert np.all(np.isfinite(x))
        np.testing.assert_array_equal(x, y)


def test_results_do_not_depend_on_host_threads():
    # the timed baseline runs on every host thread, its single-thread figure on one
    n = oracle.threads()
    toks = sm.prompt(TINY, SEED, 7)
    try:
        oracle.set_threads(1)
        assert oracle.threads() == 1
        one = _run(oracle.OracleModel(TINY, SEED), toks)
        one_pf = oracle.OracleModel(TINY, SEED).prefill(toks)
        oracle.set_threads(max(n, 3))
        many = _run(oracle.OracleModel(TINY, SEED), toks)
        many_pf = oracle.OracleModel(TINY, SEED).prefill(toks)
    finally:
        oracle.set_threads(n)
    for x, y in zip(one, many):
        np.testing.assert_array_equal(x, y)
    np.testing.assert_array_equal(one_pf, many_pf)
    np.testing.assert_array_equal(one_pf, one[-1])


def test_gqa_equals_replicated_kv_heads_model():
    """Hkv=2 model == Hkv=4 model whose k/v rows repeat each KV head twice (same Hq)."""
    cfg2 = TINY
    cfg4 = TINY.with_(n_kv_heads=4)
    d = TINY.head_dim

    def rep(l, p):
        t = sm.layer_proj(cfg2, SEED, l, p)
        if p in ("k", "v"):
            t = dict(t)
            idx = np.concatenate([np.arange(g * d, (g + 1) * d) for g in (0, 0, 1, 1)])
            t["codes"] = t["codes"][idx]
            t["scales"] = t["scales"][idx]
            t["bias"] = t["bias"][idx]
            t["N"] = 4 * d
        return t

    m2 = oracle.OracleModel(cfg2, SEED, tensors=_gen(cfg2))
    m4 = oracle.OracleModel(cfg4, SEED, tensors=rep)
    toks = sm.prompt(TINY, SEED, 5)
    for x, y in zip(_run(m2, toks), _run(m4, toks)):
        np.testing.assert_array_equal(x, y)


def test_first_position_ignores_query_and_key_weights():
    """At position 0 softmax has one entry, so q/k weights cannot matter, v weights do."""
    base = oracle.OracleModel(TINY, SEED)

    def alt(which):
        def f(l, p):
            t = sm.layer_proj(TINY, SEED, l, p)
            if p in which:
                t = dict(t)
                t["codes"] = sm.layer_proj(TINY, SEED + 1, l, p)["codes"]
            return t
        return oracle.OracleModel(TINY, SEED, tensors=f)

    tok = int(sm.prompt(TINY, SEED, 1)[0])
    ref = base.step(tok, 0)
    np.testing.assert_array_equal(alt(("q", "k")).step(tok, 0), ref)
    assert np.max(np.abs(alt(("v",)).step(tok, 0) - ref)) > 1e-3


def test_zero_layers_reduce_to_lm_head_of_normed_embedding():
    """All layer codes and biases zero: the residual stays the embedding row."""
    def zero(l, p):
        t = sm.layer_proj(TINY, SEED, l, p)
        t = dict(t)
        t["codes"] = np.zeros_like(t["codes"])
        if t["bias"] is not None:
            t["bias"] = np.zeros_like(t["bias"])
        return t

    m = oracle.OracleModel(TINY, SEED, precision="f64", tensors=zero)
    tok = 17
    logits, hidden = m.step(tok, 0, want_hidden=True)
    emb = synth.bf16_to_f32(sm.embedding(TINY, SEED)[tok]).astype(np.float64)
    np.testing.assert_array_equal(hidden, emb.astype(np.float32))
    g = synth.bf16_to_f32(sm.final_norm(TINY, SEED)).astype(np.float64)
    n = g * emb / np.sqrt(np.mean(emb ** 2) + TINY.rms_eps)
    W = synth.bf16_to_f32(sm.lm_head(TINY, SEED)["w"]).astype(np.float64)
    np.testing.assert_allclose(logits, W @ n, rtol=1e-6, atol=1e-7)


def test_mlp_hidden_permutation_invariance():
    """Permuting MLP hidden units in blocks of 128 (gate/up rows with down column groups)."""
    F = TINY.mlp
    perm_blocks = np.array([2, 0, 5, 1, 4, 3])
    assert len(perm_blocks) * 128 == F
    rows = np.concatenate([np.arange(b * 128, (b + 1) * 128) for b in perm_blocks])

    def perm(l, p):
        t = dict(sm.layer_proj(TINY, SEED, l, p))
        if p in ("gate", "up"):
            t["codes"], t["scales"] = t["codes"][rows], t["scales"][rows]
        elif p == "down":
            t["codes"], t["scales"] = t["codes"][:, rows], t["scales"][:, perm_blocks]
        return t

    a = oracle.OracleModel(TINY, SEED, precision="f64")
    b = oracle.OracleModel(TINY, SEED, precision="f64", tensors=perm)
    toks = sm.prompt(TINY, SEED, 4)
    for x, y in zip(_run(a, toks), _run(b, toks)):
        np.testing.assert_allclose(x, y, rtol=1e-6, atol=1e-6 * np.max(np.abs(x)))


def test_cache_rows_beyond_position_are_not_read():
    toks = sm.prompt(TINY, SEED, 5)
    a = oracle.OracleModel(TINY, SEED)
    ra = _run(a, toks)
    b = oracle.OracleModel(TINY, SEED)
    k, v = sm.kv_fill(TINY, 99, 0, TINY.max_context)
    for l in range(TINY.n_layers):
        b.set_kv(l, k, v)                 # garbage everywhere; each step overwrites its own row
    rb = _run(b, toks)
    for x, y in zip(ra, rb):
        np.testing.assert_array_equal(x, y)


def test_kv_cache_holds_bf16_of_rotated_keys():
    m = oracle.OracleModel(TINY, SEED, precision="f64")
    _run(m, sm.prompt(TINY, SEED, 3))
    # rows past the last position stay untouched, written rows are nonzero
    assert np.all(m.k_cache[:, 3:] == 0) and np.all(m.v_cache[:, 3:] == 0)
    assert np.all(np.any(m.k_cache[:, :3] != 0, axis=-1))


# fp32 rounding alone moves logits by ~1e-6 relative; the larger part of the gap comes
# from K/V values whose bfloat16 storage rounding flips by one ulp (2^-8 relative) between
# the two precisions.  That floor applies to any fp32 implementation, the engine included,
# and sits an order of magnitude under the 2e-2 acceptance bound.
FP32_FLOOR = 5e-3


@pytest.mark.parametrize("cfg_name", ["tiny"])
def test_fp32_variant_within_bound_of_fp64(cfg_name):
    cfg = sm.CONFIGS[cfg_name].with_(max_context=64)
    a = oracle.OracleModel(cfg, SEED, precision="f32")
    b = oracle.OracleModel(cfg, SEED, precision="f64")
    toks = sm.prompt(cfg, SEED, 12)
    for x, y in zip(_run(a, toks), _run(b, toks)):
        assert np.max(np.abs(x - y)) <= FP32_FLOOR * np.max(np.abs(y))


def test_int8_qknorm_model_runs_and_matches_fp64():
    cfg = sm.CONFIGS["qwen3-8b"].with_(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2,
                                       head_dim=64, mlp=512, vocab=512, max_context=32)
    a = oracle.OracleModel(cfg, SEED, precision="f32")
    b = oracle.OracleModel(cfg, SEED, precision="f64")
    toks = sm.prompt(cfg, SEED, 6)
    for x, y in zip(_run(a, toks), _run(b, toks)):
        assert np.all(np.isfinite(x))
        assert np.max(np.abs(x - y)) <= FP32_FLOOR * np.max(np.abs(y))


def test_qk_norm_makes_query_key_scale_irrelevant():
    """With per-head q/k RMSNorm (eps -> 0 relative), scaling q/k weight scales changes nothing."""
    cfg = sm.CONFIGS["qwen3-8b"].with_(n_layers=1, hidden=256, n_q_heads=4, n_kv_heads=2,
                                       head_dim=64, mlp=256, vocab=256, max_context=16,
                                       rms_eps=1e-12)

    def scaled(l, p):
        t = dict(sm.layer_proj(cfg, SEED, l, p))
        if p in ("q", "k"):
            t["scales"] = (t["scales"] * np.float32(4.0)).astype(np.float32)
        return t

    a = oracle.OracleModel(cfg, SEED, precision="f64")
    b = oracle.OracleModel(cfg, SEED, precision="f64", tensors=scaled)
    toks = sm.prompt(cfg, SEED, 4)
    for x, y in zip(_run(a, toks), _run(b, toks)):
        np.testing.assert_allclose(x, y, rtol=1e-6, atol=1e-6 * np.max(np.abs(x)))


# ---------------------------------------------------------------------------------------
# Pins of the composition itself: which matrix sits inside Swish, which norm feeds which
# block, and that each residual is added exactly once.  Each builds a structured special
# case through the model's tensor/norm/embedding hooks, so that a slip in the composed
# step (silu(up) * gate, the MLP fed by the attention norm or by the pre-attention
# residual, a dropped or doubled residual) changes the result.
# ["从头开始手写一个Qwen的Naive CUDA Kernel推理引擎(一)", "SwiGLU" and "RMSNorm";
#  "How To Construct Your Personal LLM Runtime From Scratch", §3 (the seven projections).]

def _bf(x):
    return synth.f32_to_bf16(np.asarray(x, np.float32))


def _f64(b):
    return synth.bf16_to_f32(b).astype(np.float64)


def _const_proj(cfg, proj, code, scale):
    N, K = sm.proj_shape(cfg, proj)
    t = dict(sm.layer_proj(cfg, SEED, 0, proj))
    t["codes"] = np.full((N, K), code, np.int8)
    t["scales"] = np.full((N, K // 128), _bf(scale), np.uint16)
    return t


def _eye_proj(cfg, proj, scale, rows=None):
    """Codes 1 on the diagonal (row i, column i) for i < min(N, K), zero elsewhere."""
    N, K = sm.proj_shape(cfg, proj)
    t = dict(sm.layer_proj(cfg, SEED, 0, proj))
    c = np.zeros((N, K), np.int8)
    n = min(N, K) if rows is None else rows
    c[np.arange(n), np.arange(n)] = 1
    t["codes"] = c
    t["scales"] = np.full((N, K // 128), _bf(scale), np.uint16)
    return t


def _edited(cfg, proj_edit=None, norm_edit=None, embed=None, precision="f64"):
    """The seeded model with some projections / norms replaced (same seed elsewhere)."""
    def tensors(l, p):
        t = dict(sm.layer_proj(cfg, SEED, l, p))
        if proj_edit and p in proj_edit:
            t = proj_edit[p](l, t)
        return t

    def norms(l):
        n = dict(sm.layer_norms(cfg, SEED, l))
        if norm_edit:
            n = norm_edit(l, n)
        return n

    return oracle.OracleModel(cfg, SEED, precision=precision, tensors=tensors, norms=norms,
                              embed=embed)


def _zero_codes(l, t):
    t = dict(t)
    t["codes"] = np.zeros_like(t["codes"])
    return t


def _const_embed(cfg, tok, value):
    e = sm.embedding(cfg, SEED).copy()
    e[tok] = _bf(np.full(cfg.hidden, value))
    return e


def test_gate_is_the_matrix_inside_swish():
    """Gate pre-activations ~ -1000 and up ~ +900: silu(gate) * up is exactly 0, so the
    MLP adds nothing and the logits equal those of the model with zero down codes.  With
    the two matrices exchanged, silu(up) * gate is ~ -1e6 and the logits move."""
    tok = 11
    emb = _const_embed(TINY, tok, 0.5)          # positive, constant residual row
    neg = lambda l, t: _const_proj(TINY, "gate", -8, 0.5)   # noqa: E731
    pos = lambda l, t: _const_proj(TINY, "up", 7, 0.5)      # noqa: E731
    base = {"o": _zero_codes, "gate": neg, "up": pos}      # residual stays the embedding row
    ref = _edited(TINY, dict(base, down=_zero_codes), embed=emb).step(tok, 0)
    got = _edited(TINY, base, embed=emb).step(tok, 0)
    np.testing.assert_array_equal(got, ref)
    swapped = {"o": _zero_codes, "gate": lambda l, t: _const_proj(TINY, "gate", 7, 0.5),
               "up": lambda l, t: _const_proj(TINY, "up", -8, 0.5)}
    moved = _edited(TINY, swapped, embed=emb).step(tok, 0)
    assert np.max(np.abs(moved - ref)) > 0.1 * np.max(np.abs(ref))


def test_mlp_is_fed_by_the_mlp_norm():
    """mlp_norm gains 0: the MLP input is exactly 0, so the MLP adds silu(0) * 0 = 0 and the
    logits equal the zero-down-codes model; the attention norm's gains stay nonzero, so an
    MLP fed by the attention norm's output would add a nonzero term."""
    toks = sm.prompt(TINY, SEED, 4)

    def zero_mlp_norm(l, n):
        n = dict(n)
        n["mlp_norm"] = np.zeros_like(n["mlp_norm"])
        return n

    a = _run(_edited(TINY, norm_edit=zero_mlp_norm), toks)
    b = _run(_edited(TINY, {"down": _zero_codes}, norm_edit=zero_mlp_norm), toks)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    # and the MLP does contribute when the gains are the seeded ones
    c = _run(_edited(TINY), toks)
    assert np.max(np.abs(c[-1] - b[-1])) > 1e-3 * np.max(np.abs(b[-1]))


def test_qkv_are_fed_by_the_attention_norm():
    """attn_norm gains 0: q, k, v reduce to their biases at every position, so the q/k/v
    codes cannot matter; the MLP norm's gains stay nonzero."""
    toks = sm.prompt(TINY, SEED, 5)

    def zero_attn_norm(l, n):
        n = dict(n)
        n["attn_norm"] = np.zeros_like(n["attn_norm"])
        return n

    other = lambda l, t: dict(t, codes=sm.layer_proj(TINY, SEED + 7, l, "q")["codes"]  # noqa
                              [: t["codes"].shape[0]])
    a = _run(_edited(TINY, norm_edit=zero_attn_norm), toks)
    b = _run(_edited(TINY, {"q": _zero_codes, "k": _zero_codes, "v": _zero_codes},
                     norm_edit=zero_attn_norm), toks)
    c = _run(_edited(TINY, {"q": other, "k": other, "v": other}, norm_edit=zero_attn_norm), toks)
    for x, y, z in zip(a, b, c):
        np.testing.assert_array_equal(x, y)
        np.testing.assert_array_equal(x, z)


def test_attention_reaches_the_residual_only_through_o_proj():
    """W_o codes 0: the final residual is the embedding plus the MLP terms alone, so new
    q/k/v weights change nothing (no attention output leaks into the residual)."""
    toks = sm.prompt(TINY, SEED, 5)
    other = lambda l, t: dict(t, codes=sm.layer_proj(TINY, SEED + 3, l, "k")["codes"]  # noqa
                              [: t["codes"].shape[0]])
    ma = _edited(TINY, {"o": _zero_codes})
    mb = _edited(TINY, {"o": _zero_codes, "q": other, "k": other, "v": other})
    for pos, t in enumerate(toks):
        la, ha = ma.step(int(t), pos, want_hidden=True)
        lb, hb = mb.step(int(t), pos, want_hidden=True)
        np.testing.assert_array_equal(ha, hb)
        np.testing.assert_array_equal(la, lb)


def _closed_form_residual(cfg, v_bias, mlp_gain, emb_row, s_gate, s_up):
    """The residual after every layer of the structured model below, in float64:
    at position 0 softmax has one entry, so head h's output is its KV group's v, which with
    zero v codes is the bf16 bias; W_o is the identity; gate and up are s_gate I and s_up I
    on the first h MLP units (zero elsewhere) and down is the identity on them."""
    x = emb_row.copy()
    G = cfg.n_q_heads // cfg.n_kv_heads
    d = cfg.head_dim
    for l in range(cfg.n_layers):
        vb = _f64(v_bias[l]).reshape(cfg.n_kv_heads, d)
        o = np.concatenate([vb[h // G] for h in range(cfg.n_q_heads)])
        x = x + o
        n2 = _f64(mlp_gain[l]) * x / np.sqrt(np.mean(x * x) + np.float64(np.float32(cfg.rms_eps)))
        g, u = s_gate * n2, s_up * n2
        x = x + g / (1.0 + np.exp(-g)) * u
    return x


def test_composed_step_matches_closed_form_special_case():
    """Structured weights make the whole step a closed form (float64, position 0):
    residual x <- x + o (o = v bias of each head's KV group, identity W_o), then
    x <- x + silu(s_g n2) * s_u n2 with n2 = RMSNorm(x) under the MLP gains, per layer; logits =
    W_lm RMSNorm(x) under the final gains.  A dropped or doubled residual, the MLP reading the
    pre-attention residual or the attention norm, swapped gate/up (s_g != s_u), or a wrong
    head-to-group map each changes the result."""
    cfg = TINY
    h, F = cfg.hidden, cfg.mlp
    assert F >= h
    s_g, s_u = 2.0, 0.5
    edits = {
        "v": _zero_codes,
        "o": lambda l, t: _eye_proj(cfg, "o", 1.0),
        "gate": lambda l, t: _eye_proj(cfg, "gate", s_g),
        "up": lambda l, t: _eye_proj(cfg, "up", s_u),
        "down": lambda l, t: _eye_proj(cfg, "down", 1.0),
    }
    m = _edited(cfg, edits)
    tok = 23
    logits, hidden = m.step(tok, 0, want_hidden=True)
    v_bias = [sm.layer_proj(cfg, SEED, l, "v")["bias"] for l in range(cfg.n_layers)]
    norms = [sm.layer_norms(cfg, SEED, l) for l in range(cfg.n_layers)]
    emb_row = _f64(sm.embedding(cfg, SEED)[tok])
    want = _closed_form_residual(cfg, v_bias, [n["mlp_norm"] for n in norms], emb_row, s_g, s_u)
    np.testing.assert_allclose(hidden, want.astype(np.float32), rtol=1e-6, atol=1e-9)
    gf = _f64(sm.final_norm(cfg, SEED))
    xf = hidden.astype(np.float64)
    nf = gf * xf / np.sqrt(np.mean(xf * xf) + np.float64(np.float32(cfg.rms_eps)))
    W = _f64(sm.lm_head(cfg, SEED)["w"])
    np.testing.assert_allclose(logits, W @ nf, rtol=1e-6, atol=1e-6 * np.max(np.abs(W @ nf)))
    # the plausible slips, evaluated on the same closed form, are far from the oracle:
    slips = {
        "swapped gate/up": _closed_form_residual(cfg, v_bias, [n["mlp_norm"] for n in norms],
                                                 emb_row, s_u, s_g),
    }
    for name, alt in slips.items():
        assert np.max(np.abs(alt - want)) > 1e-3 * np.max(np.abs(want)), name


@pytest.mark.parametrize("cfg_name,precision", [("tiny", "f32"), ("tiny", "f64"), ("q3", "f32")])
def test_prefill_equals_sequential_steps_bitwise(cfg_name, precision):
    """The multi-row prefill is the step with its loops interchanged: same logits of the last
    token and the same bf16 K/V rows, bit for bit, including a prompt that continues a cache."""
    if cfg_name == "q3":
        cfg = sm.CONFIGS["qwen3-8b"].with_(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2,
                                           head_dim=64, mlp=384, vocab=512, max_context=96)
    else:
        cfg = TINY.with_(max_context=96)
    toks = sm.prompt(cfg, SEED, 53)
    a = oracle.OracleModel(cfg, SEED, precision=precision)
    b = oracle.OracleModel(cfg, SEED, precision=precision)
    for pos, t in enumerate(toks[:37]):
        ra = a.step(int(t), pos)
    rb = b.prefill(toks[:37])
    np.testing.assert_array_equal(ra, rb)
    for pos in range(37, 53):
        ra = a.step(int(toks[pos]), pos)
    rb = b.prefill(toks[37:53], pos0=37)
    np.testing.assert_array_equal(ra, rb)
    np.testing.assert_array_equal(a.k_cache, b.k_cache)
    np.testing.assert_array_equal(a.v_cache, b.v_cache)
