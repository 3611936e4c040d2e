"""Build libattn.so (and its debug twin libattn_debug.so) in-tree with nvcc for sm_103a.

Each (head_dim, dtype, causal / split-KV) instantiation of the kernel is
compiled as its own object in parallel, then linked with the merge kernel and
the C-ABI layer into
``exact_attention_53_gb300/libattn.so``.  ``libattn_debug.so`` holds one forward
instantiation compiled with ``ATTN_DEBUG_FAULTS`` (1 ms waits and a hook that
makes one work unit's waits run out) for the failure-detection tests; the
release library never contains it.  Objects go to ``_build/`` beside this
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
DEBUG_LIB = os.path.join(PKG, "libattn_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Host code is compiled with hidden visibility: each library exports its C ABI
# (declared under a default-visibility pragma) and nothing else, so two of
# them in one process never share template code or its static state.
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I" + INCLUDE, "-I" + CSRC]

# (head_dim, bf16, causal, split): every masked/unmasked kernel, plus the
# split-KV variant of full attention.
INSTANCES = ([(d, bf16, causal, 0) for d in (64, 128, 256) for bf16 in (0, 1) for causal in (0, 1)]
             + [(d, bf16, 0, 1) for d in (64, 128, 256) for bf16 in (0, 1)])
# (head_dim, bf16, causal) of the backward
BWD_INSTANCES = [(d, bf16, causal) for d in (64, 128, 256) for bf16 in (0, 1) for causal in (0, 1)]


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
    debug_obj = os.path.join(BUILD, "attn_debug.o")
    if _stale(debug_obj, deps):
        steps.append([nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, "attn_debug.cu"), "-o",
                      debug_obj])
    if steps:
        if verbose:
            print(f"[build] compiling {len(steps)} objects with {jobs} jobs", file=sys.stderr)
        with ThreadPoolExecutor(jobs) as ex:
            list(ex.map(_run, steps))
    for lib, lib_objs in ((LIB, objs), (DEBUG_LIB, [debug_obj])):
        if _stale(lib, lib_objs):
            tmp = lib + ".tmp"
            _run([nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *lib_objs, "-o", tmp])
            os.replace(tmp, lib)
            if verbose:
                print(f"[build] linked {lib}", file=sys.stderr)
    return LIB


def _strip_params(name: str) -> str:
    """A demangled signature without its parameter list and leading return type."""
    depth = 0
    for i, ch in enumerate(name):
        if ch == "<":
            depth += 1
        elif ch == ">":
            depth -= 1
        elif ch == "(" and depth == 0 and i > 0 and name[i - 1] in ">_abcdefghijklmnopqrstuvwxyz0123456789":
            name = name[:i]
            break
    return name[5:] if name.startswith("void ") else name


def resources(jobs: int | None = None) -> str:
    """Compile every kernel instantiation with ``-Xptxas -v`` (into a scratch folder) and
    return a markdown table of what ptxas reports per entry function: registers per thread at
    launch, named barriers, stack frame and spill bytes."""
    import re
    import tempfile

    nvcc = _nvcc()
    jobs = jobs or max(1, min(len(INSTANCES) + len(BWD_INSTANCES), os.cpu_count() or 4))
    with tempfile.TemporaryDirectory() as tmp:
        cmds = []
        for d, bf16, causal, split in INSTANCES:
            cmds.append([nvcc, *ARCH, *FLAGS, "-Xptxas", "-v", f"-DATTN_D={d}",
                         f"-DATTN_BF16={bf16}", f"-DATTN_CAUSAL={causal}", f"-DATTN_SPLIT={split}",
                         "-c", os.path.join(CSRC, "attn_inst.cu"),
                         "-o", os.path.join(tmp, f"f{len(cmds)}.o")])
        for d, bf16, causal in BWD_INSTANCES:
            cmds.append([nvcc, *ARCH, *FLAGS, "-Xptxas", "-v", f"-DATTN_D={d}",
                         f"-DATTN_BF16={bf16}", f"-DATTN_CAUSAL={causal}", "-c",
                         os.path.join(CSRC, "attn_bwd_inst.cu"),
                         "-o", os.path.join(tmp, f"b{len(cmds)}.o")])
        for name in ("attn_combine", "attn_probe"):
            cmds.append([nvcc, *ARCH, *FLAGS, "-Xptxas", "-v", "-c",
                         os.path.join(CSRC, f"{name}.cu"), "-o", os.path.join(tmp, f"{name}.o")])

        def one(cmd):
            r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
            if r.returncode != 0:
                raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout)
            return r.stdout

        with ThreadPoolExecutor(jobs) as ex:
            logs = list(ex.map(one, cmds))
    rows = {}
    for log in logs:
        entry = None
        for line in log.splitlines():
            m = re.search(r"Compiling entry function '([^']+)'", line)
            if m:
                entry = m.group(1)
                rows.setdefault(entry, {})
                continue
            if entry is None:
                continue
            m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads",
                          line)
            if m:
                rows[entry].update(stack=m.group(1), spill_st=m.group(2), spill_ld=m.group(3))
            m = re.search(r"Used (\d+) registers(?:, used (\d+) barriers)?", line)
            if m:
                rows[entry].update(regs=m.group(1), barriers=m.group(2) or "0")
    names = list(rows)
    filt = shutil.which("cu++filt") or shutil.which("c++filt")
    if filt:
        out = subprocess.run([filt], input="\n".join(names), stdout=subprocess.PIPE, text=True)
        pretty = out.stdout.splitlines()
        if len(pretty) == len(names):
            names_map = dict(zip(names, pretty))
        else:
            names_map = {n: n for n in names}
    else:
        names_map = {n: n for n in names}
    lines = ["| kernel | registers/thread at launch | barriers | stack B | spill stores B | "
             "spill loads B |", "|---|---|---|---|---|---|"]
    for n in sorted(rows, key=lambda x: names_map[x]):
        r = rows[n]
        sig = _strip_params(names_map[n])
        lines.append(f"| `{sig}` | {r.get('regs', '?')} | {r.get('barriers', '?')} | "
                     f"{r.get('stack', '?')} | {r.get('spill_st', '?')} | {r.get('spill_ld', '?')} |")
    return "\n".join(lines)


if __name__ == "__main__":
    if "--resources" in sys.argv[1:]:
        print(resources())
    else:
        build(verbose=True)
