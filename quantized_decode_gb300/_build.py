"""Build libllm.so (the engine's C ABI) in-tree with nvcc for sm_103a.

Each translation unit compiles in its own process so the build stays within a minute or
two; objects go to quantized_decode_gb300/_build/ and the library next to this file.
"""
import hashlib
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
              "model_file.cu", "k_mlp.cu", "k_batch.cu", "batch.cu"]
CPP_SOURCES = ["pack.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libllm.so")
    return cand


BASE_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fopenmp",
              "--expt-relaxed-constexpr"]
ID_FILE = LIB + ".buildid"


def source_hash(extra_flags=()):
    """SHA-256 (first 16 hex digits) of every source, public header and compile flag of the
    library.  It is compiled into libllm.so (llm_build_id) and checked when the library is
    loaded, so a binary built from other sources is never used."""
    h = hashlib.sha256()
    files = sorted(os.listdir(CSRC))
    for f in files:
        h.update(f.encode() + b"\0")
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    for f in ("llm.h", "llm_ops.h"):
        with open(os.path.join(HERE, "..", "include", f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    h.update(" ".join([*ARCH, *BASE_FLAGS, *extra_flags]).encode())
    return h.hexdigest()[:16]


def build(force=False, verbose=False, extra_flags=()):
    """Compile every CUDA/C++ source and link libllm.so; returns the library path.  An
    existing library is reused only if it was built from exactly these sources and flags."""
    bid = source_hash(extra_flags)
    if not force and os.path.exists(LIB) and os.path.exists(ID_FILE):
        with open(ID_FILE) as fh:
            if fh.read().strip() == bid:
                return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    common = [*BASE_FLAGS, *extra_flags, f"-DQD_BUILD_ID=\"{bid}\""]
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
    with open(ID_FILE + ".tmp", "w") as fh:
        fh.write(bid + "\n")
    os.replace(ID_FILE + ".tmp", ID_FILE)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
