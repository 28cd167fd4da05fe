"""Host logic of bench.py (CPU): the roofline's algorithmic bytes against the sizes of the
tensors the packer actually produces, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

from synth import model as sm

from .test_model_file import TINY8, _expected_tensors

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    sys.path.insert(0, ROOT)
    import bench as b
    return b


@pytest.mark.parametrize("cfg", [sm.CONFIGS["tiny"], TINY8], ids=["int4", "int8"])
def test_algorithmic_bytes_match_the_packed_tensors(bench, cfg):
    """Per step: every packed tensor once, except the embedding (one row), plus the K/V read at
    length T and the appended row."""
    import quantized_decode_gb300 as qd
    qd.build()
    sizes = dict((n, len(b)) for n, b in _expected_tensors(cfg, 1))
    weights = sum(sizes.values()) - sizes["embed"] + cfg.hidden * 2
    T = 200
    kv = cfg.n_layers * (2 * cfg.n_kv_heads * cfg.head_dim * 2 * (T + 1))
    assert bench.algorithmic_bytes(cfg, T) == weights + kv


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--ctx", "256", "--cycle", "16", "--steps", "2",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = [l for l in out.stdout.splitlines() if l.startswith("{")][-1]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["unit"] == "ms/token" and d["higher_is_better"] is False
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 0
    assert d["fits_in_driver_run"] is True and d["steps_requested"] == 2
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "ms/token", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("cfg", [sm.CONFIGS["tiny"], TINY8], ids=["int4", "int8"])
def test_batch_bytes_reads_weights_once(bench, cfg):
    """One sequence costs what the single-sequence step does; each further sequence adds only
    its own K/V (read at its length, plus the appended row)."""
    T = 300
    assert bench.batch_bytes(cfg, [T]) == bench.algorithmic_bytes(cfg, T)
    rkv = cfg.n_kv_heads * cfg.head_dim
    kv = lambda t: cfg.n_layers * 2 * rkv * 2 * (t + 1)  # noqa: E731
    assert bench.batch_bytes(cfg, [T, 17, 40]) == bench.algorithmic_bytes(cfg, T) + kv(17) + kv(40)


@pytest.mark.parametrize("name", ["tiny", "qwen2.5-7b", "qwen3-8b"])
def test_prefill_gemm_shapes_cover_every_linear_weight(bench, name):
    """The four prefill GEMMs of a layer (QKV stacked, gate and up as one) multiply every linear
    weight of the layer exactly once."""
    cfg = sm.CONFIGS[name]
    q, kv = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    weights = cfg.hidden * (q + 2 * kv) + q * cfg.hidden + 3 * cfg.mlp * cfg.hidden
    shapes = bench.prefill_gemm_shapes(cfg)
    assert [s[0] for s in shapes] == ["qkv", "o_proj", "gate_up", "down"]
    assert sum(n * k for _, n, k in shapes) == weights
    assert all(n % 128 == 0 and k % 128 == 0 for _, n, k in shapes)
