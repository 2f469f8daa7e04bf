"""Build the package's CUDA libraries in-tree with nvcc (sm_103a only).

libq4.so      the decode-step kernels and their C ABI (include/q4.h)
libq4synth.so the seeded synthetic-input filler (kept apart from libq4.so)
Objects compile in parallel; the result lands in weight_streaming_q4_gb300/_build/.
"""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, *ARCH]

LIBS = {
    "libq4.so": ["q4_engine.cu", "q4_tc_engine.cu", "q4_bt_engine.cu", "q4_oneshot.cu", "q4_mma.cu", "q4_glue.cu", "q4_attn.cu", "q4_attn_cluster.cu", "q4_aux.cu", "q4_api.cu", "q4_noalloc.cu"],
    "libq4synth.so": ["synth.cu"],
}


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stderr


def lib_path(name: str = "libq4.so") -> str:
    return os.path.join(OUT, name)


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> dict:
    """Compile every library that is missing or older than its sources; returns their paths."""
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "q4.h"))
    jobs = []
    for lib, srcs in LIBS.items():
        for s in srcs:
            src = os.path.join(CSRC, s)
            obj = os.path.join(OUT, s.replace(".cu", ".o"))
            if force or _stale(obj, [src, *headers]):
                jobs.append([nvcc, *NVCC_FLAGS, "-c", src, "-o", obj])
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for log in ex.map(_run, jobs):
            if verbose and log:
                print(log)
    out = {}
    for lib, srcs in LIBS.items():
        objs = [os.path.join(OUT, s.replace(".cu", ".o")) for s in srcs]
        target = lib_path(lib)
        if force or _stale(target, objs):
            _run([nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", target + ".tmp"])
            os.replace(target + ".tmp", target)
        out[lib] = target
    return out


if __name__ == "__main__":
    for k, v in build(verbose=True).items():
        print(k, v)


def build_timeline(force: bool = False) -> str:
    """The timeline build of libq4.so (libq4_tl.so: the engine stamps the GPU's
    global timer at every phase, read with q4_timeline_read)."""
    out_dir = os.path.join(OUT, "timeline")
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "q4.h"))
    jobs, objs = [], []
    for s in LIBS["libq4.so"]:
        src = os.path.join(CSRC, s)
        obj = os.path.join(out_dir, s.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src, *headers]):
            jobs.append([nvcc, *NVCC_FLAGS, "-DQ4_TIMELINE", "-c", src, "-o", obj])
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(_run, jobs))
    target = os.path.join(out_dir, "libq4_tl.so")
    if force or _stale(target, objs):
        _run([nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", target + ".tmp"])
        os.replace(target + ".tmp", target)
    return target
