#!/usr/bin/env python
"""Benchmark: batch-1 INT4 decode of the Qwen2.5-Coder-7B shape at KV length ~4096.

One step = one decode token through the whole hot path (embedding, 28 x [RMSNorm+QKV+RoPE+
paged append, split-K attention + combine, o_proj + residual, RMSNorm + gate/up + SiLU*mul,
down + residual], final RMSNorm + LM head + argmax), replayed from one CUDA graph.

Inputs are seeded synthetic weights of the 7B shape (INT4 group-128, bf16 scales) resident in
HBM before timing, and a KV cache pre-filled with seeded N(0,1) bf16 values through the page
table; timed positions cycle through [ctx - cycle, ctx) so every step attends to ~ctx tokens.
The 4.7 GB read per step is far larger than L2 (129 MB), so no flush is needed between steps.

--impl reference times the CPU oracle instead: the whole 28-layer model with the real
vocabulary, greedy steps on the same seeded weights and KV fill (no extrapolation; the step
count is capped by a time budget and the steps actually run are reported).  Under torchrun
every rank runs its own replica (no collective on the data path); rank 0 prints one JSON line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 decode ms/token & HBM GB/s (7B INT4, ctx 4096); TTFT pp512"
NOMINAL_HBM_GBS = 8000.0
# DRAM bytes read + written per launch come from an ncu capture summarised in
# profiles/: lines "traffic: build=<id> shape=<name> kernel=<k> bytes=<n>".  A
# line counts only while the library's build id (a hash of every source) is the
# one it was measured on, so a changed kernel reports traffic null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic_7b.md")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
ORACLE_BUDGET_S = 240.0   # bound on the oracle's timed steps (reference arm)


def ncu_traffic(build_id, shape, kernel):
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if not line.startswith("traffic:"):
                    continue
                kv = dict(t.split("=", 1) for t in line.split()[1:] if "=" in t)
                if kv.get("build") == build_id and kv.get("shape") == shape and kv.get("kernel") == kernel:
                    return int(kv["bytes"])
    except OSError:
        pass
    return None


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=600)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default="qwen2.5-7b")
    p.add_argument("--ctx", type=int, default=4096)
    p.add_argument("--cycle", type=int, default=128, help="positions cycle in [ctx-cycle, ctx)")
    p.add_argument("--layers", type=int, default=0, help="override layer count (profiling cases)")
    p.add_argument("--vocab", type=int, default=0, help="override vocab (profiling cases)")
    p.add_argument("--seed", type=int, default=4242)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-oracle-timings", action="store_true",
                   help="skip the oracle's prefill and one-thread figures beside its baseline")
    p.add_argument("--no-ttft", action="store_true")
    p.add_argument("--ttft-only", action="store_true",
                   help="time the pp512 prefill only and print {'ttft_ms': ...} (profiling case)")
    p.add_argument("--no-variants", action="store_true",
                   help="skip the persistent / no-PDL / fused / eager comparisons (profiling case)")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-kv-sweep", action="store_true",
                   help="skip the ms/token sweep over KV lengths (512, 2048; 8192-32768 long context)")
    p.add_argument("--profile-steps", type=int, default=4)
    p.add_argument("--step", default="chain", choices=["chain", "persistent"],
                   help="decode step as a kernel chain or as one persistent kernel")
    p.add_argument("--timeline-steps", type=int, default=16,
                   help="steps of the in-graph per-kernel timeline (0: skip)")
    p.add_argument("--no-batch", action="store_true", help="skip the 8-sequence decode line")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the 1.5B (pp512/tg128) and Qwen3-8B INT8 (inputs 128..4096) lines")
    return p.parse_args()


def max_over_ranks(x, device):
    """The largest x (one float) over all ranks of the process group; x itself without one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def model_cfg(args):
    from synth import model as sm
    cfg = sm.CONFIGS[args.config]
    over = {"max_context": args.ctx}
    if args.layers:
        over["n_layers"] = args.layers
    if args.vocab:
        over["vocab"] = args.vocab
    return cfg.with_(**over)


def algorithmic_bytes(cfg, T):
    """Bytes one decode step must move at KV length T (T cached tokens incl. the new one)."""
    h, d, F, L, V = cfg.hidden, cfg.head_dim, cfg.mlp, cfg.n_layers, cfg.vocab
    rq, rkv = cfg.n_q_heads * d, cfg.n_kv_heads * d
    shapes = [(rq, h), (rkv, h), (rkv, h), (h, rq), (F, h), (F, h), (h, F)]
    per_layer = 0
    for N, K in shapes:
        if cfg.weight_format == 1:
            per_layer += N * K // 2 + N * (K // 128) * 2
        else:
            per_layer += N * K + N * 4
    if cfg.qkv_bias:
        per_layer += (rq + 2 * rkv) * 2
    per_layer += 2 * h * 2 + (2 * d * 2 if cfg.qk_norm else 0)
    kv_read = 2 * rkv * 2 * T
    kv_write = 2 * rkv * 2
    lm = V * h * (2 if (cfg.weight_format == 1 or cfg.tied_lm_head) else 1) + \
        (V * 4 if cfg.weight_format == 2 and not cfg.tied_lm_head else 0)
    return L * (per_layer + kv_read + kv_write) + lm + h * 2 + h * 2


def kernel_bytes(cfg, T):
    """Algorithmic bytes per launch of each kernel kind (for the roofline of one kernel)."""
    h, d, F, V = cfg.hidden, cfg.head_dim, cfg.mlp, cfg.vocab
    rq, rkv = cfg.n_q_heads * d, cfg.n_kv_heads * d

    def w(N, K):
        return N * K // 2 + N * (K // 128) * 2 if cfg.weight_format == 1 else N * K + N * 4

    return {
        "qkv": w(rq + 2 * rkv, h) + h * 4 + (rq + 2 * rkv) * 2 + 2 * rkv * 2 + rq * 4,
        "attention": 2 * rkv * 2 * T + rq * 4 * 2,
        "o_proj": w(h, rq) + rq * 4 + h * 4 * 2,
        "gate_up": 2 * w(F, h) + h * 4 + F * 4,
        "down": w(h, F) + F * 4 + h * 4 * 2,
        "mlp": 3 * w(F, h) + h * 4 + h * 8,
        "lm_head": V * h * 2 + h * 4 + V * 4,
    }


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while a region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sms, maxes, reasons = [], [], set()
        window = [r for t, r in self.rows if t0 - 0.15 <= t <= t1 + 0.15] or [r for _, r in self.rows]
        for r in window:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for name, val in zip(names[1:], parts[5:9]):
                if val.lower() in ("active", "0x1", "1"):
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s burst (fp16 has the same dense rate): the peak of a GEMM timed alone."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def prefill_gemm_shapes(cfg):
    """(name, N, K) of the four GEMMs of a prefill layer (gate and up as one 2F-row GEMM)."""
    d = cfg.head_dim
    return [("qkv", (cfg.n_q_heads + 2 * cfg.n_kv_heads) * d, cfg.hidden), ("o_proj", cfg.hidden, cfg.n_q_heads * d),
            ("gate_up", 2 * cfg.mlp, cfg.hidden), ("down", cfg.hidden, cfg.mlp)]


def prefill_gemms(cfg, M=512, reps=5, batch=10):
    """The prefill GEMM (llm_op_gemm_quant: weight codes dequantized inside the tcgen05 kernel)
    at the shapes of one layer of an M-row prompt: batches of `batch` back-to-back launches timed
    with CUDA events (median over reps batches), cycling through copies of the weights and
    activations that together exceed L2, so every launch reads its operands from HBM.  Seeded
    codes, unit scales: the timing does not depend on the values.  gate/up is timed with the
    plain store epilogue (the engine's SwiGLU epilogue writes half the bytes)."""
    import torch
    from quantized_decode_gb300 import _lib
    from synth import model as sm
    lib = _lib.load()
    peak, peak_kind = measured_tensor_peak()
    int4 = cfg.weight_format == sm.FMT_INT4_G128
    fmt = 1 if int4 else 2
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    out = {}
    for name, N, K in prefill_gemm_shapes(cfg):
        per = N * K // (2 if int4 else 1) + M * K * 2
        copies = max(2, -(-300_000_000 // per))
        bufs = []
        for _ in range(copies):
            A = (torch.randn(M, K, device="cuda", generator=g) * 0.5).half()
            if int4:
                w = torch.randint(-2**31, 2**31 - 1, (N * K // 8,), dtype=torch.int32, device="cuda", generator=g)
                s_ = torch.full((N * K // 128,), 0x3C00, dtype=torch.int16, device="cuda")
            else:
                w = torch.randint(-127, 128, (N * K,), dtype=torch.int8, device="cuda", generator=g)
                s_ = torch.full((N,), 1.0 / 64, dtype=torch.float32, device="cuda")
            bufs.append((A, w, s_))
        C = torch.empty(M, N, dtype=torch.float32, device="cuda")
        it = [0]

        def run():
            A, w, s_ = bufs[it[0] % copies]
            it[0] += 1
            rc = lib.llm_op_gemm_quant(fmt, A.data_ptr(), w.data_ptr(), s_.data_ptr(), M, N, K, C.data_ptr(), None)
            if rc != 0:
                raise RuntimeError(f"llm_op_gemm_quant {name}: {rc}")
        for _ in range(3):
            run()
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(batch):
                run()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / batch)
        us = float(np.median(ts))
        tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
        out[name] = {"M": M, "N": N, "K": K, "us": round(us, 2), "tflops": round(tf, 1), "frac": round(tf / peak, 3)}
        del bufs, C
        torch.cuda.empty_cache()
    out["peak_tflops"] = peak
    out["peak_kind"] = peak_kind
    return out


# ---------------------------------------------------------------- CPU oracle

def oracle_decode(cfg, seed, T0, n_warm, n_steps, rec=None, budget_s=None):
    """The oracle (fp32, all host cores) on the whole model: the seeded weights, the KV
    cache filled with the same seeded values as the GPU run up to T0, then greedy steps at
    positions T0, T0 + 1, ...  Returns (mean ms/step, sample text, steps timed)."""
    import oracle
    from synth import model as sm
    get_proj, get_norms, emb, fin, lm = rec if rec is not None else sm.recipe(cfg, seed)
    orc = oracle.OracleModel(cfg, seed, t_max=T0 + n_warm + n_steps + 1, tensors=get_proj,
                             norms=get_norms, embed=emb, lm_head=lm)
    for l in range(cfg.n_layers):
        k, v = sm.kv_fill(cfg, seed + 1, l, T0)
        orc.set_kv(l, k, v)
    tok, pos = 7, T0
    for _ in range(n_warm):
        tok = int(np.argmax(orc.step(tok, pos)))
        pos += 1
    times = []
    t_start = time.perf_counter()
    for i in range(n_steps):
        t0 = time.perf_counter()
        tok = int(np.argmax(orc.step(tok, pos)))
        times.append((time.perf_counter() - t0) * 1e3)
        pos += 1
        if budget_s is not None and time.perf_counter() - t_start > budget_s:
            break
    mean_ms = statistics.mean(times)
    sample = (f"oracle fp32, whole {cfg.name}-shape model ({cfg.n_layers} layers, vocab {cfg.vocab}): "
              f"{len(times)} greedy steps at KV {T0 + n_warm + 1}..{T0 + n_warm + len(times)} after "
              f"{n_warm} warm-up steps, mean {mean_ms:.1f} ms/token")
    return mean_ms, sample, len(times)


def oracle_timings(cfg7, rec7, seed):
    """The oracle's own prefill and per-thread figures, beside its decode baseline: pp512 of
    the tiny and 1.5B configurations, pp64 of the 7B shape, and one decode step of the tiny
    and 7B shapes on a single host thread (the oracle's results do not depend on the thread
    count).  Seeded prompts, fresh caches."""
    import oracle
    from synth import model as sm
    threads = oracle.threads()
    out = {"threads": threads}

    def timed_prefill(cfg, n, rec=None):
        get_proj, get_norms, emb, fin, lm = rec if rec is not None else sm.recipe(cfg, seed)
        orc = oracle.OracleModel(cfg, seed, t_max=n + 24, tensors=get_proj, norms=get_norms,
                                 embed=emb, lm_head=lm)
        toks = sm.prompt(cfg, seed + 7, n, stream=1)
        t0 = time.perf_counter()
        logits = orc.prefill(toks)
        ms = (time.perf_counter() - t0) * 1e3
        return orc, int(np.argmax(logits)), ms

    def one_thread_step(orc, tok, pos):
        oracle.set_threads(1)
        try:
            t0 = time.perf_counter()
            orc.step(tok, pos)
            return (time.perf_counter() - t0) * 1e3
        finally:
            oracle.set_threads(threads)

    tiny = sm.CONFIGS["tiny"].with_(max_context=1024)
    orc, tok, ms = timed_prefill(tiny, 512)
    t0 = time.perf_counter()
    for i in range(16):
        tok = int(np.argmax(orc.step(tok, 512 + i)))
    out["tiny"] = {"pp512_ms": round(ms, 1), "decode_ms_per_token": round((time.perf_counter() - t0) * 1e3 / 16, 2),
                   "decode_ms_per_token_1_thread": round(one_thread_step(orc, tok, 528), 2)}
    del orc
    b15 = sm.CONFIGS["qwen2.5-1.5b"]
    orc, _, ms = timed_prefill(b15, 512)
    out["qwen2.5-1.5b"] = {"pp512_ms": round(ms, 1)}
    del orc
    orc, tok, ms = timed_prefill(cfg7, 64, rec7)
    out[cfg7.name] = {"pp64_ms": round(ms, 1), "decode_ms_per_token_1_thread": round(one_thread_step(orc, tok, 64), 1)}
    del orc
    return out


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    cfg = model_cfg(args)
    ctx, cycle = args.ctx, min(args.cycle, args.ctx - 1)
    T0 = ctx - cycle
    n_warm = args.warmup
    t0 = time.perf_counter()
    mean_ms, sample, n_run = oracle_decode(cfg, args.seed, T0, n_warm, args.steps, budget_s=ORACLE_BUDGET_S)
    wall = time.perf_counter() - t0
    import oracle
    cores = oracle.threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(mean_ms, 3), "unit": "ms/token",
        "n_gpus": args.gpus, "steps": n_run, "steps_requested": args.steps, "warmup": n_warm,
        "ms_per_step": round(mean_ms, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded weights and KV fill)",
        "config": {"workload": f"{cfg.name}-shape INT4 g128 decode, batch 1, greedy, KV {T0 + 1}.."
                               f"{T0 + n_warm + n_run}, seeded KV", "global_batch": 1, "seq_len": ctx,
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": round(mean_ms, 3), "unit": "ms/token", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(mean_ms, 3), "unit": "ms/token", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 1),
        # every requested step ran inside the oracle's time bound (so the driver's clock
        # around this run covers the region the value claims)
        "fits_in_driver_run": n_run == args.steps,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    from quantized_decode_gb300 import DeviceModel, Engine, LLMError
    from synth import model as sm

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    cfg = model_cfg(args)
    ctx, cycle = args.ctx, min(args.cycle, args.ctx - 1)
    T0 = ctx - cycle

    t_setup = time.perf_counter()
    rec = sm.recipe(cfg, args.seed)
    model = DeviceModel(cfg, *rec)
    stream = torch.cuda.Stream()
    eng = Engine(model, stream=stream.cuda_stream)
    if args.step == "persistent":
        eng.set_persistent(True)
    setup_s = time.perf_counter() - t_setup

    # ---- TTFT pp512 (prompt of seeded uniform token ids)
    ttft_ms = None
    if not args.no_ttft:
        prompt = sm.prompt(cfg, args.seed, min(512, ctx - 1))
        eng.reset()
        eng.prefill(prompt[:8])          # warm the prefill path
        runs = []
        for _ in range(3):
            eng.reset()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            eng.prefill(prompt)
            runs.append((time.perf_counter() - t0) * 1e3)
        ttft_ms = float(np.median(runs))
        eng.reset()
    pf_gemms = None
    if not args.no_ttft and rank == 0:
        pf_gemms = prefill_gemms(cfg)
    if args.ttft_only:
        if rank == 0:
            print(json.dumps({"ttft_ms": None if ttft_ms is None else round(ttft_ms, 2), "prefill_gemms": pf_gemms}))
        eng.close()
        return

    # ---- KV filled with seeded values through a shuffled page table
    from quantized_decode_gb300.kvfill import write_kv
    import synth

    def fill_kv(e, c, seed, T, page_perm):
        write_kv(e, c, lambda l: sm.kv_fill(c, seed, l, T), T, page_perm)

    n_pages = (ctx + 15) // 16
    fill_kv(eng, cfg, args.seed + 1, T0, page_perm=synth.permutation(args.seed, 3, n_pages))

    def enqueue(n):
        """n greedy steps, rewinding to T0 whenever the next step would pass ctx."""
        launched = 0
        while n > 0:
            room = ctx - eng.seq_len()
            if room <= 0:
                eng.truncate(T0)
                launched += 1
                room = ctx - T0
            k = min(n, room)
            eng.decode_enqueue(k)
            n -= k
        return launched

    eng.decode_step(7)                       # a token to feed the greedy chain
    enqueue(args.warmup)
    eng.sync()

    # ---- timed region: graph replays, inputs resident
    start_ev = torch.cuda.Event(enable_timing=True)
    end_ev = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clk:
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        w0 = clk.mark()
        start_ev.record(stream)
        extra = enqueue(args.steps)
        end_ev.record(stream)
        torch.cuda.synchronize()
        w1 = clk.mark()
        if ws > 1:
            torch.distributed.barrier()
    eng.sync()
    elapsed_ms = start_ev.elapsed_time(end_ev)
    elapsed_ms = max_over_ranks(elapsed_ms, "cuda")
    ms_per_token = elapsed_ms / args.steps
    clocks = clk.summary(w0, w1)

    # KV lengths attended during the timed steps (cycle through [T0+1, ctx])
    mean_T = T0 + (cycle + 1) / 2.0
    step_bytes = algorithmic_bytes(cfg, mean_T)
    step_gbs = step_bytes / (ms_per_token * 1e-3) / 1e9
    peak, peak_kind = measured_peak()

    # ---- ms/token at other KV lengths of the same cache (the workload's 512 / 2048 / 4096 sweep)
    def timed_at(e, L, n=64):
        e.debug_kv(set_len=L)        # K/V rows below L hold the seeded fill (or earlier steps)
        e.decode_enqueue(4)
        e.debug_kv(set_len=L)
        s5, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s5.record(stream)
        e.decode_enqueue(n)
        e5.record(stream)
        torch.cuda.synchronize()
        e.sync()
        return round(s5.elapsed_time(e5) / n, 4)

    kv_sweep = None
    if not args.no_kv_sweep and ws == 1 and ctx >= 2048 + 64:
        kv_sweep = {str(L): timed_at(eng, L) for L in (512, 2048) if L + 64 <= ctx}
        kv_sweep[str(ctx)] = round(ms_per_token, 4)
        eng.debug_kv(set_len=T0)

    # ---- long-context decode: the same weights with a 32K cache pre-filled with seeded K/V
    # through a shuffled page table; 64 greedy steps at 8192, 16384 and 32768 tokens
    long_ctx = None
    if not args.no_kv_sweep and ws == 1 and args.layers == 0 and args.vocab == 0:
        lmax = 32768
        cfg_l = cfg.with_(max_context=lmax + 128)
        eng_l = Engine(DeviceModel(cfg_l, *rec), stream=stream.cuda_stream)
        try:
            fill_kv(eng_l, cfg_l, args.seed + 2, lmax,
                    page_perm=synth.permutation(args.seed, 4, (cfg_l.max_context + 15) // 16))
            eng_l.decode_step(7)
            long_ctx = {str(L): timed_at(eng_l, L) for L in (8192, 16384, 32768)}
        finally:
            eng_l.close()

    other_ms = no_pdl_ms = fused_ms = eager_ms = sampling_ms = act8_ms = ofold_ms = None
    if not args.no_variants:
        # ---- graph replay with o_proj, gate/up and down on int8 activations (opt-in, INT4 models)
        try:
            eng.set_act_int8(True)
            enqueue(3)
            s8, e8 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s8.record(stream)
            enqueue(100)
            e8.record(stream)
            torch.cuda.synchronize()
            act8_ms = round(s8.elapsed_time(e8) / 100, 4)
            eng.set_act_int8(False)
        except LLMError:
            pass

        # ---- graph replay with top-k / top-p sampling (Qwen's recommended 0.6 / 20 / 0.95) instead of argmax
        eng.set_sampling(0.6, 20, 0.95, args.seed)
        enqueue(3)
        s7, e7 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s7.record(stream)
        enqueue(100)
        e7.record(stream)
        torch.cuda.synchronize()
        sampling_ms = round(s7.elapsed_time(e7) / 100, 4)
        eng.set_sampling(0.0)

        # ---- the other step form (persistent kernel vs kernel chain), same cache and greedy chain
        other_ms = None
        try:
            eng.set_persistent(args.step != "persistent")
            s4, e4 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            enqueue(10)
            s4.record(stream)
            enqueue(100)
            e4.record(stream)
            torch.cuda.synchronize()
            other_ms = s4.elapsed_time(e4) / 100
        except LLMError:
            pass
        eng.set_persistent(args.step == "persistent")

        # ---- graph replay without programmatic dependent launch (the default uses it)
        eng.set_pdl(False)
        s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_pdl = 100
        s3.record(stream)
        enqueue(n_pdl)
        e3.record(stream)
        torch.cuda.synchronize()
        no_pdl_ms = s3.elapsed_time(e3) / n_pdl
        eng.set_pdl(True)

        # ---- graph replay with the fused QKV + attention kernel (opt-in, where the model fits it)
        fused_ms = None
        try:
            eng.set_fused_attention(True)
            enqueue(3)
            s6, e6 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s6.record(stream)
            enqueue(n_pdl)
            e6.record(stream)
            torch.cuda.synchronize()
            fused_ms = round(s6.elapsed_time(e6) / n_pdl, 4)
            eng.set_fused_attention(False)
        except LLMError:
            pass

        # ---- graph replay with o_proj folded into the attention clusters (the other setting of
        # llm_set_o_fold, where the attention plan allows it)
        try:
            fold_default = eng.o_fold()
            eng.set_o_fold(not fold_default)
            enqueue(3)
            s9, e9 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s9.record(stream)
            enqueue(n_pdl)
            e9.record(stream)
            torch.cuda.synchronize()
            ofold_ms = {"o_fold": not fold_default, "ms_per_token": round(s9.elapsed_time(e9) / n_pdl, 4)}
            eng.set_o_fold(fold_default)
        except LLMError:
            pass

        # ---- eager launches, same kernels (graph vs eager)
        eng.set_graph_mode(False)
        eng.sync()
        torch.cuda.synchronize()
        n_eager = 20
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        enqueue(n_eager)
        e2.record(stream)
        torch.cuda.synchronize()
        eager_ms = s2.elapsed_time(e2) / n_eager
        eng.set_graph_mode(True)

    step_kinds = eng.step_kinds() or ["step"]   # the launches of one step (persistent: one kernel)
    # ---- per-kernel share of the step inside graph replay: every launch records the time its
    # last CTA finished; launch j's share is the time from launch j-1's finish to its own
    # (the kernels overlap under programmatic dependent launch, so this partition of the step
    # period is what each kernel adds to the token's latency)
    names = ["qkv", "attention", "o_proj", "gate_up", "down"]
    kb = kernel_bytes(cfg, mean_T)
    timeline = None
    if args.timeline_steps > 1 and args.step == "chain":
        if eng.seq_len() + args.timeline_steps > ctx:
            eng.truncate(T0)
        st = eng.timeline_steps(args.timeline_steps).astype(np.int64)
        prev = np.concatenate([st[:-1, -1:], st[1:, :-1]], axis=1)      # steps 1.. only
        dur_us = (st[1:] - prev) / 1e3                                    # [steps-1][launches]
        kinds = eng.step_kinds()
        period_us = float(np.mean((st[1:, -1] - st[:-1, -1]) / 1e3))
        tl_kern = {}
        for k in dict.fromkeys(kinds):
            cols = [j for j, kk in enumerate(kinds) if kk == k]
            per_launch = dur_us[:, cols]
            tot = float(np.mean(per_launch.sum(axis=1)))
            ent = {"avg_us": round(float(np.mean(per_launch)), 2), "share": round(tot / period_us, 4)}
            if k in kb:
                ent["gbs"] = round(kb[k] / (float(np.mean(per_launch)) * 1e-6) / 1e9, 1)
            tl_kern[k] = ent
        timeline = {"steps": args.timeline_steps - 1, "period_us": round(period_us, 2), "kernels": tl_kern}

    # ---- per-kernel breakdown (events between serialised launches; secondary)
    per = {n: [] for n in names + ["lm_head"]}
    for _ in range(args.profile_steps):
        if eng.seq_len() >= ctx:
            eng.truncate(T0)
        ms = eng.profile_step()
        for l in range(cfg.n_layers):
            for j, n in enumerate(names):
                per[n].append(float(ms[5 * l + j]))
        per["lm_head"].append(float(ms[-1]))
    if all(v == 0.0 for v in per["attention"]):  # the fused QKV + attention kernel fills the QKV entry
        per = {("qkv_attention" if n == "qkv" else n): v for n, v in per.items() if n != "attention"}
        kb["qkv_attention"] = kb["qkv"] + kb["attention"]
    totals = {n: sum(v) / args.profile_steps for n, v in per.items()}
    if timeline is not None:     # the roofline of the kernel with the largest in-graph share
        dom = max((k for k in timeline["kernels"] if k in kb), key=lambda k: timeline["kernels"][k]["share"])
        avg_ms = timeline["kernels"][dom]["avg_us"] * 1e-3
        roof_src = "in-graph timeline (last-CTA finish times, graph replay with PDL)"
    else:
        dom = max(totals, key=totals.get)
        avg_ms = statistics.mean(per[dom])
        roof_src = "CUDA events between serialised launches"
    achieved = kb[dom] / (avg_ms * 1e-3) / 1e9
    breakdown = {n: {"avg_us": round(1e3 * statistics.mean(v), 2),
                     "share": round(totals[n] / sum(totals.values()), 4),
                     "gbs": round(kb[n] / (statistics.mean(v) * 1e-3) / 1e9, 1)} for n, v in per.items()}

    # ---- the other configurations' own protocols (1.5B pp512 / tg128; Qwen3-8B INT8 inputs
    # 128 .. 4096 with 128 greedy output tokens), on their own seeded models
    sweep = None
    if not args.no_sweep and ws == 1 and args.layers == 0 and args.vocab == 0:
        sweep = config_sweep(args, stream, peak, peak_kind)

    # ---- multi-sequence decode: 8 sequences of the same model over one paged pool, each step
    # reading the weights once for all of them
    batch8 = None
    if not args.no_batch and ws == 1:
        batch8 = batch_decode(args, model, cfg, stream, peak, peak_kind)

    # ---- end to end through the C ABI: host token in (pinned H2D), host token out (D2H)
    toks = sm.prompt(cfg, args.seed, args.e2e_steps, stream=1)
    if eng.seq_len() + args.e2e_steps > ctx:
        eng.truncate(max(0, ctx - args.e2e_steps - 1))
        eng.sync()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for t in toks:
        eng.decode_step(int(t))
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps

    # ---- CPU oracle baseline (rank 0, one GPU only): the whole model, a few greedy steps
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        mean_ms, sample, _ = oracle_decode(cfg, args.seed, T0, 1, 6, rec=rec)
        cpu = {"value": round(mean_ms, 2), "unit": "ms/token", "cores": oracle.threads(),
               "kind": "oracle", "sample": sample}
        if not args.no_oracle_timings:
            cpu["more"] = oracle_timings(cfg, rec, args.seed)

    tok_s = 1e3 / ms_per_token
    line = {
        "metric": METRIC, "value": round(ms_per_token, 4), "unit": "ms/token",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_token, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4 weights, fp16 products, fp32 accumulate",
        "data": "synthetic (seeded weights, prompts and KV fill)",
        "config": {"workload": f"{cfg.name}-shape INT4 g128 decode, batch 1, greedy, KV {T0 + 1}..{ctx} "
                               f"(mean {mean_T:.0f}), seeded KV through a shuffled page table",
                   "global_batch": 1, "seq_len": ctx, "parallelism": "replicas" if ws > 1 else "single",
                   "l2": "inputs larger than L2 (4.7 GB per step vs 129 MB)"},
        "tokens_per_s": round(tok_s * ws, 2),
        "hbm_gbs": round(step_gbs, 1),
        "step_roofline": {"bound": "hbm", "achieved": round(step_gbs, 1), "peak": peak,
                          "unit": "GB/s", "frac": round(step_gbs / peak, 4), "peak_kind": peak_kind,
                          "frac_of_8tbs": round(step_gbs / NOMINAL_HBM_GBS, 4),
                          "bytes_per_step": int(step_bytes)},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": ncu_traffic(eng.lib.llm_build_id().decode(), cfg.name, dom),
                     "bytes_per_launch": int(kb[dom]), "avg_launch_us": round(avg_ms * 1e3, 2),
                     "peak_kind": peak_kind, "duration_source": roof_src},
        "kernels_in_graph": timeline,
        "kernels_serialised": breakdown,
        "ttft_ms": None if ttft_ms is None else round(ttft_ms, 2),
        "prefill_gemms": pf_gemms,
        "kv_sweep_ms_per_token": kv_sweep,
        "long_context_ms_per_token": long_ctx,
        "eager_ms_per_token": None if eager_ms is None else round(eager_ms, 4),
        "graph_no_pdl_ms_per_token": None if no_pdl_ms is None else round(no_pdl_ms, 4),
        "fused_qkv_attention_ms_per_token": fused_ms,
        "o_fold_other_setting": ofold_ms,
        "sampling_ms_per_token": sampling_ms,
        "act_int8_ms_per_token": act8_ms,
        ("chain_ms_per_token" if args.step == "persistent" else "persistent_ms_per_token"):
            None if other_ms is None else round(other_ms, 4),
        "config_sweep": sweep,
        "batch_decode": batch8,
        "e2e": {"value": round(e2e_ms, 4), "unit": "ms/token", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 8},
        "gpu_launches": args.steps * len(step_kinds) + extra,
        "clocks": clocks,
        "setup_s": round(setup_s, 1),
    }
    if cpu:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    eng.close()
    if ws > 1:
        torch.distributed.destroy_process_group()


def batch_bytes(cfg, lengths):
    """Bytes one multi-sequence step must move: every weight once, plus each sequence's K/V
    read at its length and its appended row."""
    rkv = cfg.n_kv_heads * cfg.head_dim
    one = algorithmic_bytes(cfg, 0) - cfg.n_layers * 2 * rkv * 2   # weights (+ embedding row)
    return one + sum(cfg.n_layers * (2 * rkv * 2 * (T + 1)) for T in lengths)


def batch_decode(args, model, cfg, stream, peak, peak_kind, B=8, prompt_len=64, n=64):
    """tok/s of B sequences decoding together (llm_batch_step), after a prompt each."""
    from quantized_decode_gb300 import BatchEngine
    from synth import model as sm
    eng = BatchEngine(model, B, stream=stream.cuda_stream, config=None)
    try:
        seqs = [eng.add() for _ in range(B)]
        for s in seqs:
            eng.prefill(s, sm.prompt(cfg, args.seed + 100 + s, prompt_len, stream=100 + s))
        for _ in range(3):
            eng.step(seqs)
        t0 = time.perf_counter()
        for _ in range(n):
            eng.step(seqs)
        dt = (time.perf_counter() - t0) / n
        lengths = [prompt_len + 3 + n / 2] * B
        gbs = batch_bytes(cfg, lengths) / dt / 1e9
        return {"sequences": B, "ms_per_step": round(dt * 1e3, 3), "tokens_per_s": round(B / dt, 1),
                "step_roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                  "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                                  "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)},
                "timing": "wall clock around llm_batch_step (host page allocation and copies included)",
                "kv_len_mean": prompt_len + 3 + n / 2}
    finally:
        eng.close()


def config_sweep(args, stream, peak, peak_kind):
    """TTFT and decode ms/token of the 1.5B (pp512 / tg128) and Qwen3-8B INT8 (inputs
    128 .. 4096, 128 greedy output tokens each) configurations, graph replay, seeded inputs."""
    import torch
    from quantized_decode_gb300 import DeviceModel, Engine
    from synth import model as sm

    def decode_ms(eng, n):
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        eng.decode_enqueue(n)
        e0.record(stream)
        torch.cuda.synchronize()
        eng.sync()
        return s0.elapsed_time(e0) / n

    def roof(cfg, T, ms):
        gbs = algorithmic_bytes(cfg, T) / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4), "kv_len_mean": T}

    out = {}
    # Qwen2.5-1.5B shape: 512-token prompt, then 128 greedy tokens
    cfg = sm.CONFIGS["qwen2.5-1.5b"].with_(max_context=1024)
    eng = Engine(DeviceModel(cfg, *sm.recipe(cfg, args.seed)), stream=stream.cuda_stream)
    try:
        prompt = sm.prompt(cfg, args.seed, 512)
        eng.prefill(prompt[:8])
        ttft = []
        for _ in range(3):
            eng.reset()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            eng.prefill(prompt)
            ttft.append((time.perf_counter() - t0) * 1e3)
        eng.decode_enqueue(3)                       # warm-up
        eng.sync()
        eng.truncate(513)
        ms = decode_ms(eng, 128)
        out[cfg.name] = {"ttft_pp512_ms": round(float(np.median(ttft)), 2), "tg128_ms_per_token": round(ms, 4),
                         "tokens_per_s": round(1e3 / ms, 1), "step_roofline": roof(cfg, 512 + 64.5, ms)}
    finally:
        eng.close()
    # Qwen3-8B shape, INT8 per-row weights and LM head: inputs 128 .. 4096, 128 output tokens
    cfg = sm.CONFIGS["qwen3-8b"]
    eng = Engine(DeviceModel(cfg, *sm.recipe(cfg, args.seed)), stream=stream.cuda_stream)
    try:
        per_input, ttft = {}, {}
        for n_in in (128, 512, 1024, 2048, 4096):
            prompt = sm.prompt(cfg, args.seed, n_in)
            eng.reset()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            eng.prefill(prompt)
            ttft[str(n_in)] = round((time.perf_counter() - t0) * 1e3, 2)
            per_input[str(n_in)] = round(decode_ms(eng, 128), 4)
        out[cfg.name] = {"tpot_ms_by_input": per_input, "ttft_ms_by_input": ttft,
                         "step_roofline_input_4096": roof(cfg, 4096 + 64.5, per_input["4096"]),
                         "step_roofline_input_128": roof(cfg, 128 + 64.5, per_input["128"])}
    finally:
        eng.close()
    return out


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
