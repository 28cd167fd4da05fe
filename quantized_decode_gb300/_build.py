"""Build libllm.so (the engine's C ABI) in-tree with nvcc for sm_103a.

Each translation unit compiles in its own process so the build stays within a minute or
two; objects go to quantized_decode_gb300/_build/ and the library next to this file.
"""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libllm.so")

CU_SOURCES = ["engine.cu", "ops.cu", "ops_noalloc.cu", "k_qkv.cu", "k_gemv.cu", "k_lmhead.cu",
              "k_attn.cu", "k_qkv_attn.cu", "k_sample.cu", "k_step.cu", "k_tcgemm.cu", "k_prefill.cu",
              "model_file.cu"]
CPP_SOURCES = ["pack.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libllm.so")
    return cand


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(HERE, "..", "include", f) for f in ("llm.h", "llm_ops.h")]
    return max(os.path.getmtime(f) for f in files if os.path.exists(f))


def build(force=False, verbose=False, extra_flags=()):
    """Compile every CUDA/C++ source and link libllm.so; returns the library path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps() and not extra_flags:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    common = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fopenmp",
              "--expt-relaxed-constexpr", *extra_flags]
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmd = [nvcc, *ARCH, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for src in CPP_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-fopenmp", "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose and text:
            sys.stdout.write(f"--- {src}\n{text}")
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"libllm.so build failed:\n{msg}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fopenmp"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
