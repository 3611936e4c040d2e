"""Build libattn.so in-tree with nvcc for sm_103a.

Each (head_dim, dtype, causal / split-KV) instantiation of the kernel is
compiled as its own object in parallel, then linked with the merge kernel and
the C-ABI layer into
``exact_attention_53_gb300/libattn.so``.  Objects go to ``_build/`` beside this
file; an object is rebuilt only when a source or header is newer than it.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]

# (head_dim, bf16, causal, split): every masked/unmasked kernel, plus the
# split-KV variant of full attention.
INSTANCES = ([(d, bf16, causal, 0) for d in (64, 128, 256) for bf16 in (0, 1) for causal in (0, 1)]
             + [(d, bf16, 0, 1) for d in (64, 128, 256) for bf16 in (0, 1)])
# (head_dim, bf16, causal) of the backward
BWD_INSTANCES = [(d, bf16, causal) for d in (64, 128) for bf16 in (0, 1) for causal in (0, 1)]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin on PATH)")


def _deps() -> list[str]:
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)
            if f.endswith((".cu", ".cuh", ".h"))] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout)


def build(verbose: bool = False, jobs: int | None = None) -> str:
    """Compile and link libattn.so if anything changed; return its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    deps = _deps()
    jobs = jobs or max(1, min(len(INSTANCES) + len(BWD_INSTANCES) + 4, os.cpu_count() or 4))
    steps = []
    objs = []
    for d, bf16, causal, split in INSTANCES:
        mode = "split" if split else ("causal" if causal else "full")
        obj = os.path.join(BUILD, f"attn_fwd_d{d}_{'bf16' if bf16 else 'f16'}_{mode}.o")
        objs.append(obj)
        if _stale(obj, deps):
            steps.append([nvcc, *ARCH, *FLAGS, f"-DATTN_D={d}", f"-DATTN_BF16={bf16}",
                          f"-DATTN_CAUSAL={causal}", f"-DATTN_SPLIT={split}", "-c",
                          os.path.join(CSRC, "attn_inst.cu"), "-o", obj])
    for d, bf16, causal in BWD_INSTANCES:
        obj = os.path.join(BUILD, f"attn_bwd_d{d}_{'bf16' if bf16 else 'f16'}_{'causal' if causal else 'full'}.o")
        objs.append(obj)
        if _stale(obj, deps):
            steps.append([nvcc, *ARCH, *FLAGS, f"-DATTN_D={d}", f"-DATTN_BF16={bf16}",
                          f"-DATTN_CAUSAL={causal}", "-c", os.path.join(CSRC, "attn_bwd_inst.cu"),
                          "-o", obj])
    for name in ("attn_api", "attn_combine", "attn_noalloc", "attn_probe"):
        obj = os.path.join(BUILD, f"{name}.o")
        objs.append(obj)
        if _stale(obj, deps):
            steps.append([nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, f"{name}.cu"), "-o", obj])
    if steps:
        if verbose:
            print(f"[build] compiling {len(steps)} objects with {jobs} jobs", file=sys.stderr)
        with ThreadPoolExecutor(jobs) as ex:
            list(ex.map(_run, steps))
    if steps or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp])
        os.replace(tmp, LIB)
        if verbose:
            print(f"[build] linked {LIB}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
