"""Build the CUDA libraries in-tree (nvcc, sm_103a only, no cmake).

    libsmoe.so        the C-ABI library declared in include/smoe.h
    libsmoe_synth.so  the benchmark's on-device input generator
                      (include/smoe_synth.h; no part of the method)

Translation units compile in parallel; outputs land in
``bit_expert_weight_gb300/_build/`` (git-ignored).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
           "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]

LIBS = {
    "libsmoe.so": ["api.cu", "quant.cu", "repack.cu", "router.cu", "layer.cu", "grouped.cu", "noalloc.cu",
                   "vault.cu"],
    "libsmoe_synth.so": ["synth.cu"],
}


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    inc = os.path.join(ROOT, "include")
    hs += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    return hs


def _compile(src: str, log: list) -> str:
    obj = os.path.join(OUT, os.path.basename(src) + ".o")
    if _stale(obj, [src] + _headers()):
        cmd = [nvcc()] + ARCH + NVFLAGS + ["-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        log.append((src, r.stdout + r.stderr))
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False) -> dict:
    """Compile and link every library; returns {name: path}."""
    os.makedirs(OUT, exist_ok=True)
    log: list = []
    out = {}
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        futs = {lib: [ex.submit(_compile, os.path.join(CSRC, s), log) for s in srcs]
                for lib, srcs in LIBS.items()}
        for lib, fs in futs.items():
            objs = [f.result() for f in fs]
            so = os.path.join(OUT, lib)
            if _stale(so, objs):
                cmd = [nvcc()] + ARCH + ["-shared", "-o", so + ".tmp"] + objs + ["-lcudart"]
                r = subprocess.run(cmd, capture_output=True, text=True)
                if r.returncode != 0:
                    raise RuntimeError(f"link failed for {lib}:\n{r.stderr}")
                os.replace(so + ".tmp", so)
            out[lib] = so
    if verbose:
        for src, text in log:
            print(f"== {os.path.basename(src)}\n{text}")
    return out


if __name__ == "__main__":
    build(verbose=True)
